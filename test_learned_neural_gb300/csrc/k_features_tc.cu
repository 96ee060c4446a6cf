// Projected polynomial features on the tensor cores: out = phi(x) P for every
// key and query row, phi(x) = [1, x_i, x_i x_j / 2 (i <= j, lexicographic)]
// (atlas-torch README, "Atlas Extensions": Polynomial Features, projected
// back by a fixed matrix; ATLAS summary, Section 3.1).  For 64-dim keys that
// is 2145 monomials projected to 64.
//
// One CTA per SM, persistent over tiles of 128 rows.  The monomials never
// reach global memory: for each K stage of 64 monomials the CTA's 512
// threads generate the tile's 128 x 64 values from the raw rows held in
// shared memory.  Each row is extended to x' = [x, 1, 0], so every feature
// is one product x'_i x'_j (constant: 1 * 1; linear: x_i * 1; quadratic:
// x_i x_j; padding: 0 * 0) from a table of index pairs read eight at a
// time; the 1/2 of the quadratic monomials is folded into P^T (exact in
// bf16).  Each value v is stored as two bf16 parts, hi = bf16(v) and lo =
// bf16(v - hi) (about 2^-17 relative, below the rounding of the fp32 sum
// over 2145 terms), in the 128-byte-swizzled K-major layout.  P is bf16, so
// hi P + lo P (tcgen05.mma, fp32 accumulation in 64 TMEM columns) gives
// phi P to that accuracy.  P^T (transposed, halved on the quadratic rows and
// zero-padded to a multiple of 64 monomials once per call) arrives by TMA,
// two stages ahead, in a four-slot ring.  Stage s + 1 is generated while
// the MMAs of stage s run; a stage's A buffer and P slot are reused once its
// MMAs have completed (tcgen05.commit on an mbarrier).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {
namespace {

constexpr int FM = 128, FK = 64, FN = 64, NT = 512, PSLOTS = 4, AHEAD = 2;
constexpr int A_PART = FM * FK * 2;            // one bf16 part of a stage's A tile (16 KB)
constexpr int A_BUF = 2 * A_PART;              // hi, lo
constexpr int P_STAGE = FN * FK * 2;           // 8 KB
constexpr long long kWait = 1ll << 31;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(tc::smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
// K-major operand, 128-byte swizzle: 8-row groups 1024 bytes apart
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

struct FeatSmem {
  int xs, pij, abuf, pring, total;
};
__host__ __device__ inline FeatSmem feat_smem(int d) {
  FeatSmem s;
  s.abuf = 0;                                  // 2 x A_BUF, 1024-aligned
  s.pring = 2 * A_BUF;                         // PSLOTS x P_STAGE
  s.xs = s.pring + PSLOTS * P_STAGE;           // [FM][d + 3] fp32: x, 1, 0 (odd stride)
  s.pij = s.xs + (FM * (d + 3) * 4 + 15) / 16 * 16;   // [Kpad] uint16 pair index (i << 8 | j)
  s.total = s.pij;                             // + Kpad * 2, added by the host
  return s;
}

__global__ void __launch_bounds__(NT, 1) k_features_proj_tc(Geom g, const void* __restrict__ src,
                                                           const void* __restrict__ cache, int rows_per_unit,
                                                           int from_cache, const __grid_constant__ CUtensorMap map_pt,
                                                           int Kpad, float* __restrict__ out, int* status) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int d = g.d_k, ld = d + 3;
  const FeatSmem L = feat_smem(d);
  float* xs = reinterpret_cast<float*>(sm + L.xs);
  uint16_t* pij = reinterpret_cast<uint16_t*>(sm + L.pij);
  __shared__ uint64_t full[PSLOTS], abar[2], done;
  __shared__ uint32_t tbase;
  __shared__ int failed;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const long long total_rows = (long long)g.units * rows_per_unit;
  const int ntiles = (int)((total_rows + FM - 1) / FM);
  const int nk = Kpad / FK;
  const int mytiles = blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const long long mystages = (long long)mytiles * nk;

  if (warp == 0) tc::tmem_alloc(&tbase, FN);
  if (tid == 0) {
    for (int s = 0; s < PSLOTS; ++s) tc::mbar_init(&full[s], 1);
    tc::mbar_init(&abar[0], 1);
    tc::mbar_init(&abar[1], 1);
    tc::mbar_init(&done, 1);
    failed = 0;
  }
  // feature f = x'_i x'_j with x' = [x, 1 (column d), 0 (column d + 1)]:
  // constant (d, d), linear (f - 1, d), quadratic (i, j), i <= j in
  // lexicographic order, padding (d + 1, d + 1)
  for (int f = tid; f < Kpad; f += NT) {
    int i, j;
    if (f == 0) { i = d; j = d; }
    else if (f <= d) { i = f - 1; j = d; }
    else if (f < g.poly) {
      int q = f - 1 - d;
      i = 0;
      while (q >= d - i) { q -= d - i; ++i; }
      j = i + q;
    } else { i = d + 1; j = d + 1; }
    pij[f] = (uint16_t)((i << 8) | j);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tacc = tbase;
  const uint32_t idesc = tc::idesc_f16(FM, FN, 1, 0, 0);

  // P^T stage of global stage gs (the same column block in every tile)
  auto issue_p = [&](long long gs) {
    const int s = (int)(gs % PSLOTS);
    mbar_expect_tx(&full[s], P_STAGE);
    tma_load_2d(sm + L.pring + s * P_STAGE, &map_pt, (int)(gs % nk) * FK, 0, &full[s]);
  };
  if (tid == 0)
    for (long long gs = 0; gs < AHEAD && gs < mystages; ++gs) issue_p(gs);

  bool ok = true;
  long long gs = 0;   // global stage counter of this CTA
  int ti = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++ti) {
    // raw rows of the tile (cache rows first for keys) as fp32 x' = [x, 1, 0]:
    // thread = (row tid / 4, columns 16 (tid % 4) ..), one index division each
    {
      const int r = tid >> 2, k0 = (tid & 3) * 16;
      const long long R = (long long)tile * FM + r;
      float* xr = xs + r * ld;
      const uint16_t* rowp = nullptr;
      if (R < total_rows) {
        const int u = (int)(R / rows_per_unit), row = (int)(R % rows_per_unit);
        if (from_cache && row < g.n_prev)
          rowp = (const uint16_t*)cache + ((size_t)u * (g.c - 1) + (size_t)(g.c - 1 - g.n_prev + row)) * d;
        else
          rowp = (const uint16_t*)src + ((size_t)u * g.T + (row - (from_cache ? g.n_prev : 0))) * d;
      }
      for (int kb = k0; kb < d; kb += 64)
        for (int k = kb; k < kb + 16 && k < d; ++k) xr[k] = rowp ? __uint_as_float(((uint32_t)__ldg(rowp + k)) << 16) : 0.f;
      if ((tid & 3) == 0) {
        xr[d] = 1.f;
        xr[d + 1] = 0.f;
      }
    }
    __syncthreads();
    for (int kt = 0; kt < nk; ++kt, ++gs) {
      const int b = (int)(gs & 1);
      // the A buffer (and the P slot) of stage gs - 2 are free once its MMAs are done
      if (gs >= 2) ok = ok && tc::mbar_wait(&abar[b], (uint32_t)(((gs >> 1) - 1) & 1), kWait);
      if (tid == 0 && ok && gs + AHEAD < mystages) issue_p(gs + AHEAD);
      // generate: thread = (row r, 16 monomials), 2 chunks of 8
      {
        const int r = tid & (FM - 1), quarter = tid >> 7;
        uint8_t* ab = sm + L.abuf + b * A_BUF;
        const float* xr = xs + r * ld;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = 2 * quarter + c, f0 = kt * FK + 8 * chunk;
          const uint4 pp = *reinterpret_cast<const uint4*>(pij + f0);   // 8 pairs
          const uint32_t pw[4] = {pp.x, pp.y, pp.z, pp.w};
          float v[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t w2 = pw[e];
            v[2 * e] = xr[(w2 >> 8) & 255] * xr[w2 & 255];
            v[2 * e + 1] = xr[w2 >> 24] * xr[(w2 >> 16) & 255];
          }
          __nv_bfloat162 hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            const float2 h = __bfloat1622float2(hi[e]);
            lo[e] = __floats2bfloat162_rn(v[2 * e] - h.x, v[2 * e + 1] - h.y);
          }
          const int off = r * 128 + ((chunk ^ (r & 7)) << 4);   // 128-byte swizzle
          *reinterpret_cast<uint4*>(ab + off) = *reinterpret_cast<const uint4*>(hi);
          *reinterpret_cast<uint4*>(ab + A_PART + off) = *reinterpret_cast<const uint4*>(lo);
        }
      }
      tc::fence_smem_to_async();
      tc::fence_before_sync();
      if (__syncthreads_or(!ok)) ok = false;
      tc::fence_after_sync();
      if (tid == 0 && ok) {
        const int s = (int)(gs % PSLOTS);
        if (tc::mbar_wait(&full[s], (uint32_t)((gs / PSLOTS) & 1), kWait)) {
          tc::fence_after_sync();
          const uint8_t* ab = sm + L.abuf + b * A_BUF;
          const uint64_t bd0 = sdesc_sw128(tc::smem_u32(sm + L.pring + s * P_STAGE));
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint64_t ad = sdesc_sw128(tc::smem_u32(ab + p * A_PART)), bd = bd0;
#pragma unroll
            for (int ks = 0; ks < FK / 16; ++ks) {
              tc::mma_f16(tacc, ad, bd, idesc, (kt > 0 || p > 0 || ks > 0) ? 1u : 0u);
              ad += 2;   // 32 bytes along K in the swizzled row
              bd += 2;
            }
          }
          tc::mma_commit(&abar[b]);
        } else {
          atomicExch(&failed, 1);
        }
      }
    }
    // accumulator complete: read out, rows of 64 fp32 (256 contiguous bytes each)
    if (tid == 0) tc::mma_commit(&done);
    ok = ok && tc::mbar_wait(&done, (uint32_t)(ti & 1), kWait);
    if (__syncthreads_or(!ok) || failed) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    {
      // 16 warps: lane quarter q = warp % 4, 16 columns (warp / 4)
      const int q = warp & 3, c0 = 16 * (warp >> 2);
      const int r = 32 * q + lane;
      float v[16];
      tc::tmem_ld16(tacc + ((uint32_t)(32 * q) << 16) + c0, v);
      tc::tmem_ld_wait();
      const long long R = (long long)tile * FM + r;
      if (R < total_rows) {
        float* o = out + R * g.F + c0;
#pragma unroll
        for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
    }
    tc::fence_before_sync();
    __syncthreads();   // TMEM read and xs free for the next tile
    tc::fence_after_sync();
  }
  if (!ok || failed) {
    if (tid == 0) {
      // let the TMA copies in flight land before the shared memory is released
      for (int s = 0; s < PSLOTS; ++s) tc::mbar_wait(&full[s], 0, kWait / 16);
      atomicExch(status, ATLAS_ERR_TIMEOUT);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, FN);
}

// P [poly][proj] (bf16 bits) -> Pt [proj][Kpad]: zero-padded monomials,
// the quadratic rows (f > d) halved (the 1/2! of phi; exact in bf16)
__global__ void k_transpose_p(const uint16_t* __restrict__ P, uint16_t* __restrict__ Pt, int poly, int proj,
                              int Kpad, int d) {
  __shared__ uint16_t tile[32][33];
  const int f0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int f = f0 + i, j = j0 + threadIdx.x;
    uint16_t v = 0;
    if (f < poly && j < proj) {
      v = P[(size_t)f * proj + j];
      if (f > d) v = __bfloat16_as_ushort(__float2bfloat16_rn(0.5f * __uint_as_float(((uint32_t)v) << 16)));
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int j = j0 + i, f = f0 + threadIdx.x;
    if (j < proj && f < Kpad) Pt[(size_t)j * Kpad + f] = tile[threadIdx.x][i];
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

}  // namespace

int features_tc_kpad(const Geom& g) { return (g.poly + FK - 1) / FK * FK; }

// the tensor-core path: bf16 inputs and P, degree 2, 64 projected features,
// keys of at most 254 dims (pair table of x' = [x, 1, 0]), the raw rows in
// shared memory
bool features_tc_supported(const Geom& g) {
  if (!(g.proj_dim == FN && g.p == 2 && g.qkv_dtype == ATLAS_BF16 && g.d_k <= 254)) return false;
  const size_t smem = (size_t)feat_smem(g.d_k).total + (size_t)features_tc_kpad(g) * 2 + 1024;
  return smem <= 227 * 1024;
}

size_t features_tc_scratch_bytes(const Geom& g) {
  return features_tc_supported(g) ? (size_t)FN * features_tc_kpad(g) * 2 : 0;
}

// P transposed into Pt (scratch of features_tc_scratch_bytes, 16-byte aligned)
cudaError_t features_tc_prepare(const Geom& g, const void* P, void* Pt, cudaStream_t st) {
  const int Kpad = features_tc_kpad(g);
  dim3 grid((FN + 31) / 32, (Kpad + 31) / 32);
  k_transpose_p<<<grid, dim3(32, 8), 0, st>>>((const uint16_t*)P, (uint16_t*)Pt, g.poly, FN, Kpad, g.d_k);
  return cudaGetLastError();
}

cudaError_t features_tc_launch(const Geom& g, const void* src, const void* cache, int rows, int from_cache,
                               const void* Pt, float* out, int* status, cudaStream_t st) {
  const int Kpad = features_tc_kpad(g);
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)Kpad, (cuuint64_t)FN};
  const cuuint64_t strides[1] = {(cuuint64_t)Kpad * 2};
  const cuuint32_t box[2] = {FK, FN};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(Pt), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int smem = feat_smem(g.d_k).total + Kpad * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_features_proj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long total = (long long)g.units * rows;
  const int ntiles = (int)((total + FM - 1) / FM);
  const int sms = num_sms();
  const int grid = ntiles < sms ? ntiles : sms;
  if (grid <= 0) return cudaSuccess;
  k_features_proj_tc<<<grid, NT, smem, st>>>(g, src, cache, rows, from_cache, map, Kpad, out, status);
  return cudaGetLastError();
}

}  // namespace atlas
