// The projection of the stage in front of the memory, U = x W_in (x [M][D],
// W_in [D][N], U [M][Np] fp32 with the row stride padded to 16 bytes).
//
// bf16 inputs: a persistent, warp-specialised tcgen05 GEMM.  W_in is first
// transposed to W_t [N][K] (one small kernel), so both operands are K-major.
// Output tiles are 128 x 256, K = D in stages of 64; each CTA takes tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... (N fastest, so CTAs working at
// the same time share x rows in L2).
//   warp 0   TMA producer: per stage one box of 64 elements (128 bytes) x
//            128 rows per operand, in the 128-byte-swizzled layout (row r
//            at r * 128, its 16-byte chunk j at j ^ (r % 8), 8-row groups
//            1024 bytes apart), into a three-stage ring on "full" mbarriers;
//   warp 1   MMA issuer: four K = 16 steps per stage (bf16 operands, fp32
//            accumulation), descriptors with SBO = 1024 and the 128-byte
//            swizzle stepped by 32 bytes along K; commits free the stage
//            and, after a tile's last stage, hand its accumulator over;
//   warps 2-9 epilogue: two accumulators of 256 TMEM columns alternate, so
//            one tile's accumulator is read out while the next one fills;
//            two warps per TMEM lane quarter split the columns; rows go
//            through a per-warp shared-memory block and leave as coalesced
//            128-byte row segments.
// Out-of-range rows and columns read as zeros.  x and W_in are bf16, so the
// products are exact and only the fp32 accumulation rounds.
//
// fp32 inputs, or bf16 ones whose strides or addresses TMA cannot take: a
// register-tiled fp32 GEMM (64 x 64 per CTA).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/atlas_mem.h"
#include "tc.cuh"

namespace atlas {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 3, EPI_WARPS = 8, NTHR = 64 + 32 * EPI_WARPS;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BK * BN * 2, STAGE_BYTES = A_BYTES + B_BYTES;
static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
constexpr int EPI_LD = 36;                                      // staging row stride (floats)
constexpr int EPI_BYTES = EPI_WARPS * 32 * EPI_LD * 4;          // one 32 x 32 block per epilogue warp
constexpr int SMEM_TC = STAGES * STAGE_BYTES + EPI_BYTES + 1024;  // + alignment slack
constexpr long long kWaitCycles = 1ll << 31;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(tc::smem_u32(bar))
      : "memory");
}

// shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: 8-row groups SBO = 1024 bytes apart (LBO unused: the
// K extent of a stage, 64 bf16, is one swizzle row), layout type 2
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                      // LBO (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;            // SBO
  d |= (uint64_t)1 << 46;                      // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(NTHR, 1) k_proj_tc(const __grid_constant__ CUtensorMap map_x,
                                                     const __grid_constant__ CUtensorMap map_wt, int M, int N, int Np,
                                                     int K, float* __restrict__ U, int* status) {
  extern __shared__ uint8_t smraw[];
  // 1024-byte aligned ring (the swizzle pattern repeats every 1024 bytes)
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  float* epi = reinterpret_cast<float*>(sm + STAGES * STAGE_BYTES);
  __shared__ uint64_t full[STAGES], empty[STAGES], acc_full[2], acc_empty[2];
  __shared__ uint32_t tbase;
  __shared__ int failed;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int ntn = (N + BN - 1) / BN, ntiles = ntn * ((M + BM - 1) / BM);
  const int nk = (K + BK - 1) / BK;

  if (warp == 0) tc::tmem_alloc(&tbase, 2 * BN);
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 32 * EPI_WARPS);   // every epilogue thread
    }
    failed = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tacc = tbase;

  if (warp == 0) {
    if (lane == 0) {
      // producer: ring slot it % STAGES, reused once the MMAs that read it are done
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int m0 = (tile / ntn) * BM, n0 = (tile % ntn) * BN;
        for (int kt = 0; kt < nk; ++kt, ++it) {
          const int s = it % STAGES;
          if (it >= STAGES && !(ok = tc::mbar_wait(&empty[s], ((it / STAGES) - 1) & 1, kWaitCycles))) break;
          mbar_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(sm + s * STAGE_BYTES, &map_x, kt * BK, m0, &full[s]);
          tma_load_2d(sm + s * STAGE_BYTES + A_BYTES, &map_wt, kt * BK, n0, &full[s]);
        }
      }
      if (!ok) atomicExch(&failed, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(BM, BN, 1, 0, 0);
      int it = 0, i = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++i) {
        const int a = i & 1;
        // the epilogue has read this accumulator's previous tile
        if (i >= 2 && !(ok = tc::mbar_wait(&acc_empty[a], ((i >> 1) - 1) & 1, kWaitCycles))) break;
        tc::fence_after_sync();
        for (int kt = 0; kt < nk; ++kt, ++it) {
          const int s = it % STAGES;
          if (!(ok = tc::mbar_wait(&full[s], (it / STAGES) & 1, kWaitCycles))) break;
          tc::fence_after_sync();
          uint64_t ad = sdesc_sw128(tc::smem_u32(sm + s * STAGE_BYTES));
          uint64_t bd = sdesc_sw128(tc::smem_u32(sm + s * STAGE_BYTES + A_BYTES));
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            tc::mma_f16(tacc + a * BN, ad, bd, idesc, (kt > 0 || ks > 0) ? 1u : 0u);
            ad += (uint64_t)(32 >> 4);   // 16 bf16 further along K inside the swizzled row
            bd += (uint64_t)(32 >> 4);
          }
          tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&acc_full[a]);   // the tile's accumulator is complete
      }
      if (!ok) atomicExch(&failed, 1);
    }
  } else {
    // epilogue warps 2-9: TMEM lane quarter q = warp % 4 (rows 32 q ..
    // 32 q + 31), column half h (128 columns, two 64-column passes)
    const int q = warp & 3, h = (warp - 2) >> 2;
    float* blk = epi + (warp - 2) * 32 * EPI_LD;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int i = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
      const int a = i & 1;
      // warp-uniform: the tcgen05.ld below are .sync.aligned
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&acc_full[a], (i >> 1) & 1, kWaitCycles));
      if (!ok) {
        atomicExch(&failed, 1);
        break;
      }
      tc::fence_after_sync();
      const int m0 = (tile / ntn) * BM, n0 = (tile % ntn) * BN;
      // this warp's 128 columns of its 32 rows, 64 at a time, each pass's
      // TMEM loads issued before its stores
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
      float v2[2][32];
      const uint32_t cbase = tacc + a * BN + lane_base + 128 * h + 64 * pass;
      tc::tmem_ld16(cbase, v2[0]);
      tc::tmem_ld16(cbase + 16, v2[0] + 16);
      tc::tmem_ld16(cbase + 32, v2[1]);
      tc::tmem_ld16(cbase + 48, v2[1] + 16);
      tc::tmem_ld_wait();
      if (pass == 1) {
        // every TMEM read of this accumulator by this thread is done: hand it back
        tc::fence_before_sync();
        mbar_arrive(&acc_empty[a]);
      }
#pragma unroll
      for (int cc2 = 0; cc2 < 2; ++cc2) {
        const int c0 = 128 * h + 64 * pass + 32 * cc2;
        const float* v = v2[cc2];
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(blk + lane * EPI_LD + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        __syncwarp();
        // rows of the block: 8 lanes x 16 bytes per row, 4 rows per step
        const int rr = lane >> 3, cc = (lane & 7) * 4, col = n0 + c0 + cc;
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 4) {
          const int m = m0 + 32 * q + r0 + rr;
          if (m < M && col < Np)
            *reinterpret_cast<float4*>(U + (size_t)m * Np + col) =
                *reinterpret_cast<const float4*>(blk + (r0 + rr) * EPI_LD + cc);
        }
        __syncwarp();
      }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (failed && tid == 0) {
    // let every copy this CTA issued land before its memory is freed
    for (int s = 0; s < STAGES; ++s) tc::mbar_wait(&empty[s], 0, kWaitCycles / 16);
    atomicExch(status, ATLAS_ERR_TIMEOUT);
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 2 * BN);
}

// W [K][N] -> Wt [N][K] (bf16 bit patterns), 32 x 32 tiles
__global__ void k_transpose_bf16(const uint16_t* __restrict__ W, uint16_t* __restrict__ Wt, int K, int N) {
  __shared__ uint16_t tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int k = k0 + i, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[i][threadIdx.x] = W[(size_t)k * N + n];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int n = n0 + i, k = k0 + threadIdx.x;
    if (n < N && k < K) Wt[(size_t)n * K + k] = tile[threadIdx.x][i];
  }
}

// fp32 fallback: 64 x 64 tile per CTA, 16 x 16 threads with 4 x 4 outputs
template <typename TIn>
__device__ __forceinline__ float ldin(const TIn* p, size_t i);
template <>
__device__ __forceinline__ float ldin<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldin<uint16_t>(const uint16_t* p, size_t i) {
  return __uint_as_float(((uint32_t)p[i]) << 16);
}

template <typename TIn>
__global__ void __launch_bounds__(256) k_proj_simt(const TIn* __restrict__ x, const TIn* __restrict__ W, int M, int N,
                                                   int Np, int K, float* __restrict__ U) {
  __shared__ float As[16][68], Bs[16][68];   // As[k][m], Bs[k][n]
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int l = threadIdx.x; l < 16 * 64; l += 256) {
      const int kk = l % 16, mm = l / 16;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? ldin<TIn>(x, (size_t)m * K + k) : 0.f;
      const int nn = l % 64, kb = l / 64;
      const int n = n0 + nn, kr = k0 + kb;
      Bs[kb][nn] = (n < N && kr < K) ? ldin<TIn>(W, (size_t)kr * N + n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < Np) U[(size_t)m * Np + n] = n < N ? acc[i][j] : 0.f;
    }
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

// 2-D bf16 tensor map over a row-major [rows][cols] array with boxes of
// 64 columns (128 bytes) x box_rows rows, 128-byte swizzled in shared memory
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Bytes of scratch the tensor-core path needs for W_t (0 if it cannot run).
size_t proj_gemm_scratch(int N, int K, int bf16) {
  return (bf16 && K % 8 == 0) ? ((size_t)N * K * 2 + 255) / 256 * 256 : 0;
}

// U [M][Np] = x [M][K] W [K][N]; wt: scratch of proj_gemm_scratch bytes
// (16-byte aligned) for W transposed.  Returns the error of the launches.
// *kind: 1 = tensor cores (TMA + tcgen05), 0 = the fp32 SIMT GEMM.
cudaError_t proj_gemm(const void* x, const void* W, int M, int N, int Np, int K, int bf16, float* U, void* wt,
                      int* status, cudaStream_t st, int* kind) {
  *kind = 0;
  // TMA needs 16-byte aligned bases and row strides (K multiple of 8)
  const bool tma_ok = bf16 && K % 8 == 0 && wt != nullptr && (reinterpret_cast<uintptr_t>(x) % 16) == 0 &&
                      (reinterpret_cast<uintptr_t>(wt) % 16) == 0 && Np % 4 == 0;
  if (tma_ok) {
    CUtensorMap mx, mw;
    if (make_map(&mx, x, (uint64_t)M, (uint64_t)K, BM) && make_map(&mw, wt, (uint64_t)N, (uint64_t)K, BN)) {
      dim3 tg((N + 31) / 32, (K + 31) / 32);
      k_transpose_bf16<<<tg, dim3(32, 8), 0, st>>>((const uint16_t*)W, (uint16_t*)wt, K, N);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k_proj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TC);
      if (e != cudaSuccess) return e;
      int dev = 0, sms = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      const int ntiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
      const int grid = ntiles < sms ? ntiles : (sms > 0 ? sms : 1);   // persistent: one CTA per SM
      k_proj_tc<<<grid, NTHR, SMEM_TC, st>>>(mx, mw, M, N, Np, K, U, status);
      *kind = 1;
      return cudaGetLastError();
    }
  }
  dim3 grid((Np + 63) / 64, (M + 63) / 64);
  if (bf16)
    k_proj_simt<uint16_t><<<grid, 256, 0, st>>>((const uint16_t*)x, (const uint16_t*)W, M, N, Np, K, U);
  else
    k_proj_simt<float><<<grid, 256, 0, st>>>((const float*)x, (const float*)W, M, N, Np, K, U);
  return cudaGetLastError();
}

}  // namespace atlas
