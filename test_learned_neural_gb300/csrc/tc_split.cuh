// Split-bf16 tensor-core products with fp32 operands staged by the kernel:
// every fp32 value x goes into two bf16 tiles, hi = bf16(x) and lo =
// bf16(x - hi) (16 significant bits together), and a product is the three
// MMAs hi hi' + hi lo' + lo hi' with fp32 accumulation in TMEM (the dropped
// lo lo' term is about 2^-18 relative).  Tiles use the no-swizzle
// core-matrix layout of tc.cuh.
#pragma once
#include <cuda_bf16.h>

#include "tc.cuh"

namespace tcs {

// 8 consecutive fp32 values -> bf16 hi and lo chunks (16 bytes each) at byte
// offset off of the two tiles
__device__ __forceinline__ void put8(uint8_t* hi, uint8_t* lo, uint32_t off, const float* v) {
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

// An operand tile pair and its descriptor strides.  K-major (rows = M or N,
// columns = K): lbo = 128, sbo = row-group stride, 256 bytes per K step of
// 16.  MN-major (rows = K, columns = M or N): lbo = row-group stride (k
// groups), sbo = 128, two row groups per K step.
struct Opnd {
  uint32_t hi, lo, lbo, sbo, kstep;
};
__device__ __forceinline__ Opnd kmajor(const uint8_t* hi, const uint8_t* lo, int rgs) {
  return Opnd{tc::smem_u32(hi), tc::smem_u32(lo), 128u, (uint32_t)rgs, 256u};
}
__device__ __forceinline__ Opnd mnmajor(const uint8_t* hi, const uint8_t* lo, int rgs) {
  return Opnd{tc::smem_u32(hi), tc::smem_u32(lo), (uint32_t)rgs, 128u, (uint32_t)(2 * rgs)};
}
// the operand shifted by `bytes` (a column or row offset inside the tiles)
__device__ __forceinline__ Opnd shifted(Opnd o, uint32_t bytes) {
  o.hi += bytes;
  o.lo += bytes;
  return o;
}

// D (+)= A B over K (a multiple of 16) in three products; one thread.
// idesc carries M, N and the operands' major-ness.
__device__ __forceinline__ void mma3(uint32_t d, const Opnd& a, const Opnd& b, uint32_t idesc, int K, bool accumulate) {
  const uint32_t as[3] = {a.hi, a.hi, a.lo}, bs[3] = {b.hi, b.lo, b.hi};
  for (int p = 0; p < 3; ++p) {
    uint64_t ad = tc::sdesc(as[p], a.lbo, a.sbo), bd = tc::sdesc(bs[p], b.lbo, b.sbo);
    for (int ks = 0; ks < K / 16; ++ks) {
      tc::mma_f16(d, ad, bd, idesc, (accumulate || p > 0 || ks > 0) ? 1u : 0u);
      ad += a.kstep >> 4;
      bd += b.kstep >> 4;
    }
  }
}

// generic-proxy shared-memory writes -> the tensor core, then a CTA barrier
__device__ __forceinline__ void sync_for_mma() {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// Commit thread 0's MMAs to *bar and wait (every thread, bounded): false on
// a timeout, which the caller records; phase flips either way.
__device__ __forceinline__ bool commit_wait(uint64_t* bar, uint32_t& phase, bool ok, long long max_cycles) {
  if (threadIdx.x == 0 && ok) tc::mma_commit(bar);
  bool good = true;
  if (ok) good = tc::mbar_wait(bar, phase, max_cycles);
  phase ^= 1;
  const bool bad = __syncthreads_or(!good);
  tc::fence_after_sync();
  return ok && !bad;
}

}  // namespace tcs
