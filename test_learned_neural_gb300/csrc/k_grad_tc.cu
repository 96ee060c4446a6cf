// Gradient factors of the residual MLP memory at the chunk-start weights, on
// the tensor cores: for the chunk's window rows x_i (i < nw <= 128),
//   z = x W1,  a = SiLU(z),  yhat = x + a W2,  dy = 2 gamma (yhat - v),
//   dz = (dy W2^T) * SiLU'(z)
// (titans-pytorch-mlx README, Eq. 12: the loss ||M(k) - v||^2; its gradient
// with respect to W1 and W2 is sum_i x_i^T dz_i and sum_i a_i^T dy_i, which
// the Newton-Schulz path assembles from these factors).
//
// Two tensor-core kernels with one CTA per (unit, 64-wide hidden block c),
// all window rows in one M = 128 tile (rows >= nw are zero), around the
// elementwise dy step of the fp32 path:
//   k_grad2_tc_fwd: Z_c = X W1[:, c] -> z, a = SiLU(z) to global;
//                   partial Yhat_c = a_c W2[c, :] to the per-block slots
//   (k_grad2_dy):   dy = 2 gamma (x + sum_c Yhat_c - v)
//   k_grad2_tc_dz:  dz_c = (dy W2[c, :]^T) * SiLU'(z_c)
// Operands are staged from fp32 with each value split into bf16 hi/lo (x =
// hi + lo, 16 significant bits); every product is hi hi' + hi lo' + lo hi'
// with fp32 accumulation in TMEM (the split the Newton-Schulz products use:
// the momentum these factors feed is orthogonalised).  Operand tiles use the
// no-swizzle core-matrix layout of tc.cuh.
#include <cuda_bf16.h>

#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {
namespace {

constexpr int GM = 128, GH = 64, GT = 256;   // rows, hidden chunk, threads
constexpr long long kWait = 1ll << 31;

// 8 consecutive fp32 values -> hi and lo bf16 chunks (16 bytes each)
__device__ __forceinline__ void split8(uint8_t* hi, uint8_t* lo, uint32_t off, const float* v) {
  __nv_bfloat162 h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    const float2 hf = __bfloat1622float2(h[i]);
    l[i] = __floats2bfloat162_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
  }
  *reinterpret_cast<uint4*>(hi + off) = *reinterpret_cast<const uint4*>(h);
  *reinterpret_cast<uint4*>(lo + off) = *reinterpret_cast<const uint4*>(l);
}

// D (+)= A B^T over K, split bf16: hi hi' + hi lo' + lo hi'.  A K-major
// [M][K] (row-group stride aK); B K-major [N][K] (b_mn = 0) or MN-major
// [K][N] (b_mn = 1), row-group stride bK.
__device__ __forceinline__ void mma3(uint32_t d, const uint8_t* a_hi, const uint8_t* a_lo, int aK, const uint8_t* b_hi,
                                     const uint8_t* b_lo, int bK, int b_mn, int M, int N, int K, bool accumulate) {
  const uint32_t idesc = tc::idesc_f16(M, N, 1, 0, b_mn);
  const uint8_t* As[3] = {a_hi, a_hi, a_lo};
  const uint8_t* Bs[3] = {b_hi, b_lo, b_hi};
  const uint64_t bstep = (uint64_t)((b_mn ? 2 * bK : 256) >> 4);
  for (int p = 0; p < 3; ++p) {
    uint64_t ad = tc::sdesc(tc::smem_u32(As[p]), 128, aK);
    uint64_t bd = b_mn ? tc::sdesc(tc::smem_u32(Bs[p]), bK, 128) : tc::sdesc(tc::smem_u32(Bs[p]), 128, bK);
    for (int ks = 0; ks < K / 16; ++ks) {
      tc::mma_f16(d, ad, bd, idesc, (accumulate || p > 0 || ks > 0) ? 1u : 0u);
      ad += 256 >> 4;
      bd += bstep;
    }
  }
}

__device__ __forceinline__ void sync_for_mma() {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// X (or dy) rows, K-major [128][d], split; fp32 source rows of stride ld
__device__ __forceinline__ void stage_rows(uint8_t* hi, uint8_t* lo, const float* src, int ld, int nw, int d) {
  const int rgsD = (d / 8) * 128;
  for (int e = threadIdx.x; e < GM * (d / 8); e += GT) {
    const int r = e / (d / 8), k0 = (e % (d / 8)) * 8;
    float v[8];
    if (r < nw) {
      const float4 a0 = *reinterpret_cast<const float4*>(src + (size_t)r * ld + k0);
      const float4 a1 = *reinterpret_cast<const float4*>(src + (size_t)r * ld + k0 + 4);
      v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w; v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    split8(hi, lo, tc::core_offset(r, k0, rgsD), v);
  }
}

struct Ctx3 {
  uint64_t* bar;
  uint32_t phase;
  bool ok;
};
__device__ __forceinline__ void commit_wait3(Ctx3& c) {
  if (threadIdx.x == 0 && c.ok) tc::mma_commit(c.bar);
  const bool good = c.ok ? tc::mbar_wait(c.bar, c.phase, kWait) : true;
  c.phase ^= 1;
  if (__syncthreads_or(!good)) c.ok = false;
  tc::fence_after_sync();
}

}  // namespace

// smem: X (2 * 128 * d * 2), W1 block MN-major [d][64], W2 block MN-major
// [64][d], a block K-major [128][64], each hi + lo
__host__ __device__ inline int grad_fwd_smem(int d) { return 2 * GM * d * 2 + 2 * d * GH * 2 + 2 * GH * d * 2 + 2 * GM * GH * 2; }
// smem: dy (2 * 128 * d * 2), W2 block K-major [64][d]
__host__ __device__ inline int grad_dz_smem(int d) { return 2 * GM * d * 2 + 2 * GH * d * 2; }

__global__ void __launch_bounds__(GT, 1) k_grad2_tc_fwd(Geom g, Chunk ch, Work w, int buf, float* part) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int c = blockIdx.x, u = blockIdx.y, d = g.d_v, h = g.hidden, nw = ch.nw, nb = h / GH;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int q = warp & 3, half = warp >> 2, row = 32 * q + lane;   // TMEM lane = row
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  uint8_t* x_hi = sm;
  uint8_t* x_lo = x_hi + GM * d * 2;
  uint8_t* w1_hi = x_lo + GM * d * 2;
  uint8_t* w1_lo = w1_hi + d * GH * 2;
  uint8_t* w2_hi = w1_lo + d * GH * 2;
  uint8_t* w2_lo = w2_hi + GH * d * 2;
  uint8_t* a_hi = w2_lo + GH * d * 2;
  uint8_t* a_lo = a_hi + GM * GH * 2;
  const int rgsD = (d / 8) * 128, rgsH = (GH / 8) * 128;
  const float* Xw = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
  const float* W1 = w.Wst[buf][0] + (size_t)u * g.F * h;
  const float* W2 = w.Wst[buf][1] + (size_t)u * h * d;

  if (warp == 0) tc::tmem_alloc(&tbase, 256);
  if (tid == 0) tc::mbar_init(&bar, 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tZ = tbase, tY = tbase + 64;
  Ctx3 cx{&bar, 0u, true};

  stage_rows(x_hi, x_lo, Xw, g.F, nw, d);
  // W1[:, 64c ..] as MN-major B ([K = d][N = 64]); W2[64c .., :] as MN-major
  // B of a W2 ([K = 64][N = d])
  for (int e = tid; e < d * (GH / 8); e += GT) {
    const int k = e / (GH / 8), n0 = (e % (GH / 8)) * 8;
    const float* src = W1 + (size_t)k * h + GH * c + n0;
    float v[8];
    *reinterpret_cast<float4*>(v) = *reinterpret_cast<const float4*>(src);
    *reinterpret_cast<float4*>(v + 4) = *reinterpret_cast<const float4*>(src + 4);
    split8(w1_hi, w1_lo, tc::core_offset(k, n0, rgsH), v);
  }
  for (int e = tid; e < GH * (d / 8); e += GT) {
    const int k = e / (d / 8), n0 = (e % (d / 8)) * 8;
    const float* src = W2 + (size_t)(GH * c + k) * d + n0;
    float v[8];
    *reinterpret_cast<float4*>(v) = *reinterpret_cast<const float4*>(src);
    *reinterpret_cast<float4*>(v + 4) = *reinterpret_cast<const float4*>(src + 4);
    split8(w2_hi, w2_lo, tc::core_offset(k, n0, rgsD), v);
  }
  sync_for_mma();
  if (tid == 0 && cx.ok) mma3(tZ, x_hi, x_lo, rgsD, w1_hi, w1_lo, rgsH, 1, GM, GH, d, false);
  commit_wait3(cx);
  if (cx.ok) {
    // z, a = SiLU(z) of my row, block columns 32 half .. + 32
    float z[32];
    tc::tmem_ld16(tZ + lane_base + 32 * half, z);
    tc::tmem_ld16(tZ + lane_base + 32 * half + 16, z + 16);
    tc::tmem_ld_wait();
    float a[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = siluf_(z[i]);
    if (row < nw) {
      const size_t o = ((size_t)u * g.Kw + row) * h + GH * c + 32 * half;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        *reinterpret_cast<float4*>(w.Zpre + o + i) = make_float4(z[i], z[i + 1], z[i + 2], z[i + 3]);
        *reinterpret_cast<float4*>(w.Aact + o + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; j += 8) split8(a_hi, a_lo, tc::core_offset(row, 32 * half + j, rgsH), a + j);
  }
  sync_for_mma();
  if (tid == 0 && cx.ok) mma3(tY, a_hi, a_lo, rgsH, w2_hi, w2_lo, rgsD, 1, GM, d, GH, false);
  commit_wait3(cx);
  if (cx.ok) {
    // this block's partial Yhat: my row, d / 2 columns.  tcgen05.ld is
    // warp-wide (.sync.aligned): every lane loads, only rows < nw store.
    const int cw = d / 2;
    float* o = part + (((size_t)u * nb + c) * g.Kw + row) * d + half * cw;
    for (int j0 = 0; j0 < cw; j0 += 16) {
      float yv[16];
      tc::tmem_ld16(tY + lane_base + half * cw + j0, yv);
      tc::tmem_ld_wait();
      if (row < nw) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(o + j0 + i) = make_float4(yv[i], yv[i + 1], yv[i + 2], yv[i + 3]);
      }
    }
  }
  if (!cx.ok && tid == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 256);
}

// W2s: the chunk-start W2 of every unit, [units][h][d]
__global__ void __launch_bounds__(GT, 1) k_grad2_tc_dz(Geom g, Chunk ch, Work w, const float* __restrict__ W2s) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int c = blockIdx.x, u = blockIdx.y, d = g.d_v, h = g.hidden, nw = ch.nw;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int q = warp & 3, half = warp >> 2, row = 32 * q + lane;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  uint8_t* y_hi = sm;
  uint8_t* y_lo = y_hi + GM * d * 2;
  uint8_t* w_hi = y_lo + GM * d * 2;
  uint8_t* w_lo = w_hi + GH * d * 2;
  const int rgsD = (d / 8) * 128;
  if (warp == 0) tc::tmem_alloc(&tbase, 64);
  if (tid == 0) tc::mbar_init(&bar, 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  Ctx3 cx{&bar, 0u, true};
  stage_rows(y_hi, y_lo, w.DY + (size_t)u * g.Kw * d, d, nw, d);
  // W2[64c .. 64c + 64, :] as K-major B ([N = 64][K = d])
  const float* W2b = W2s + (size_t)u * h * d;
  for (int e = tid; e < GH * (d / 8); e += GT) {
    const int n = e / (d / 8), k0 = (e % (d / 8)) * 8;
    const float* src = W2b + (size_t)(GH * c + n) * d + k0;
    float v[8];
    *reinterpret_cast<float4*>(v) = *reinterpret_cast<const float4*>(src);
    *reinterpret_cast<float4*>(v + 4) = *reinterpret_cast<const float4*>(src + 4);
    split8(w_hi, w_lo, tc::core_offset(n, k0, rgsD), v);
  }
  sync_for_mma();
  if (tid == 0 && cx.ok) mma3(tbase, y_hi, y_lo, rgsD, w_hi, w_lo, rgsD, 0, GM, GH, d, false);
  commit_wait3(cx);
  if (cx.ok) {
    float t[32];
    tc::tmem_ld16(tbase + lane_base + 32 * half, t);
    tc::tmem_ld16(tbase + lane_base + 32 * half + 16, t + 16);
    tc::tmem_ld_wait();
    if (row < nw) {
      const size_t o = ((size_t)u * g.Kw + row) * h + GH * c + 32 * half;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 z4 = *reinterpret_cast<const float4*>(w.Zpre + o + i);
        *reinterpret_cast<float4*>(w.DZ + o + i) = make_float4(t[i] * dsiluf_(z4.x), t[i + 1] * dsiluf_(z4.y),
                                                               t[i + 2] * dsiluf_(z4.z), t[i + 3] * dsiluf_(z4.w));
      }
    }
  }
  if (!cx.ok && tid == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 64);
}

// depth 2, d = d_v = F in {64, 128}, hidden a multiple of 64 up to 512,
// window rows <= 128
bool grad_tc_supported(const Geom& g) {
  return g.depth == 2 && (g.d_v == 64 || g.d_v == 128) && g.F == g.d_v && g.hidden % GH == 0 && g.hidden <= 512 &&
         g.Kw <= GM && grad_fwd_smem(g.d_v) <= 227 * 1024;
}

cudaError_t grad_tc_fwd_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, float* part, cudaStream_t st) {
  const int smem = grad_fwd_smem(g.d_v);
  cudaError_t e = cudaFuncSetAttribute(k_grad2_tc_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k_grad2_tc_fwd<<<dim3(g.hidden / GH, g.units), GT, smem, st>>>(g, ch, w, buf, part);
  return cudaGetLastError();
}

cudaError_t grad_tc_dz_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, cudaStream_t st) {
  const int smem = grad_dz_smem(g.d_v);
  cudaError_t e = cudaFuncSetAttribute(k_grad2_tc_dz, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k_grad2_tc_dz<<<dim3(g.hidden / GH, g.units), GT, smem, st>>>(g, ch, w, w.Wst[buf][1]);
  return cudaGetLastError();
}

}  // namespace atlas
