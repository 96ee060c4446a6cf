// Self-test of the tensor-core building blocks (tc.cuh): one tcgen05.mma
// chain D = A * B^T from shared-memory operands in the core-matrix layout,
// dumped raw from all 128 TMEM lanes so that a test can check the
// accumulator layout for M = 64 and M = 128 against a plain matmul.
#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {

__global__ void __launch_bounds__(128) k_selftest_mma(int M, int N, int K, int a_mn, int b_mn, int bf16,
                                                      const uint16_t* A, const uint16_t* B, float* raw, int* status) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  uint8_t* As = sm;
  uint8_t* Bs = sm + (size_t)M * K * 2;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 0) tc::tmem_alloc(&tbase, 256);
  if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
  const int rgsK = (K / 8) * 128, rgsN = (N / 8) * 128, rgsM = (M / 8) * 128;
  for (int e = threadIdx.x; e < M * K; e += blockDim.x) {
    if (a_mn) *(uint16_t*)(As + tc::core_offset(e / M, e % M, rgsM)) = A[e];   // A stored [K][M]
    else *(uint16_t*)(As + tc::core_offset(e / K, e % K, rgsK)) = A[e];        // A stored [M][K]
  }
  for (int e = threadIdx.x; e < N * K; e += blockDim.x) {
    if (b_mn) *(uint16_t*)(Bs + tc::core_offset(e / N, e % N, rgsN)) = B[e];   // B stored [K][N]
    else *(uint16_t*)(Bs + tc::core_offset(e / K, e % K, rgsK)) = B[e];        // B stored [N][K]
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t d = tbase;
  if (threadIdx.x == 0) {
    const uint32_t idesc = tc::idesc_f16(M, N, bf16, a_mn, b_mn);
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ad = a_mn ? tc::sdesc(tc::smem_u32(As) + ks * 2 * rgsM, rgsM, 128)
                               : tc::sdesc(tc::smem_u32(As) + ks * 256, 128, rgsK);
      const uint64_t bd = b_mn ? tc::sdesc(tc::smem_u32(Bs) + ks * 2 * rgsN, rgsN, 128)
                               : tc::sdesc(tc::smem_u32(Bs) + ks * 256, 128, rgsK);
      tc::mma_f16(d, ad, bd, idesc, ks > 0);
    }
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0, 1ll << 30);
  tc::fence_after_sync();
  if (!ok) {
    if (threadIdx.x == 0) atomicExch(status, 1);
  } else {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tc::tmem_ld16(d + ((uint32_t)(32 * warp) << 16) + c, v);
      tc::tmem_ld_wait();
      for (int i = 0; i < 16; ++i) raw[(size_t)(32 * warp + lane) * N + c + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 256);
}

}  // namespace atlas

// Dump of the 16x32bx2 TMEM load after an M = 64 MMA: raw[(warp * 32 + t) * 16 + j]
// holds register j of thread t of warp `warp` when the warp loads columns
// [c, c + 32) of its sub-partition with a half-warp split of 16 columns.
__global__ void __launch_bounds__(128) k_selftest_ld16x2(int N, int K, const uint16_t* A, const uint16_t* B,
                                                         float* raw, int col, int* status) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int M = 64;
  uint8_t* As = sm;
  uint8_t* Bs = sm + (size_t)M * K * 2;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 0) tc::tmem_alloc(&tbase, 256);
  if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
  const int rgsK = (K / 8) * 128;
  for (int e = threadIdx.x; e < M * K; e += blockDim.x) *(uint16_t*)(As + tc::core_offset(e / K, e % K, rgsK)) = A[e];
  for (int e = threadIdx.x; e < N * K; e += blockDim.x) *(uint16_t*)(Bs + tc::core_offset(e / K, e % K, rgsK)) = B[e];
  // mark lanes 16-31 of every sub-partition over the accumulator's columns
  {
    float mark[16];
    for (int j = 0; j < 16; ++j) mark[j] = 1000.f + warp * 100 + j;
    for (int c = 0; c < N; c += 32) tc::tmem_st16_x2(tbase + ((uint32_t)(32 * warp + 16) << 16) + c, mark);
    tc::tmem_st_wait();
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (threadIdx.x == 0) {
    const uint32_t idesc = tc::idesc_f16(M, N, 1, 0, 0);
    for (int ks = 0; ks < K / 16; ++ks)
      tc::mma_f16(tbase, tc::sdesc(tc::smem_u32(As) + ks * 256, 128, rgsK),
                  tc::sdesc(tc::smem_u32(Bs) + ks * 256, 128, rgsK), idesc, ks > 0);
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0, 1ll << 30);
  tc::fence_after_sync();
  if (!ok) {
    if (threadIdx.x == 0) atomicExch(status, 1);
  } else {
    float v[16], m[16];
    tc::tmem_ld16_x2(tbase + ((uint32_t)(32 * warp) << 16) + col, v);
    tc::tmem_ld16_x2(tbase + ((uint32_t)(32 * warp + 16) << 16) + col, m);
    tc::tmem_ld_wait();
    for (int j = 0; j < 16; ++j) raw[(size_t)(warp * 32 + lane) * 16 + j] = v[j];
    // lanes 16-31 must still hold their marks after the M = 64 MMA
    for (int j = 0; j < 16; ++j)
      if (m[j] != 1000.f + warp * 100 + j) atomicExch(status, 2);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 256);
}

// A bounded mbarrier wait that runs out: the barrier expects one arrival
// and nothing arrives, so thread 0's wait (the library's own bounded wait,
// limited to max_cycles) gives up, records ATLAS_ERR_TIMEOUT in the status
// word and returns; no trap, no fault, the context stays usable.
__global__ void __launch_bounds__(32) k_selftest_timeout(long long max_cycles, int* status, long long* waited) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
  __syncthreads();
  if (threadIdx.x != 0) return;
  const long long t0 = clock64();
  const bool ok = tc::mbar_wait(&bar, 0, max_cycles);
  *waited = clock64() - t0;
  if (!ok) atomicExch(status, ATLAS_ERR_TIMEOUT);
}

extern "C" int atlas_mem_selftest_wait_timeout(long long max_cycles, int* status, long long* waited_cycles,
                                               void* stream) {
  using namespace atlas;
  if (max_cycles < 1 || max_cycles > (1ll << 31) || !status || !waited_cycles) return ATLAS_ERR_INVALID_ARG;
  k_selftest_timeout<<<1, 32, 0, (cudaStream_t)stream>>>(max_cycles, status, waited_cycles);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

extern "C" int atlas_mem_selftest_ld16x2(int N, int K, const void* A, const void* B, float* raw_out, int col,
                                         int* status, void* stream) {
  using namespace atlas;
  if (N < 64 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16 || col < 0 || col + 32 > N || !A || !B ||
      !raw_out || !status)
    return ATLAS_ERR_INVALID_ARG;
  const int smem = 200 * 1024;
  cudaFuncSetAttribute(k_selftest_ld16x2, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k_selftest_ld16x2<<<1, 128, smem, (cudaStream_t)stream>>>(N, K, (const uint16_t*)A, (const uint16_t*)B, raw_out,
                                                            col, status);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}

extern "C" int atlas_mem_selftest_mma(int M, int N, int K, int a_mn_major, int b_mn_major, int bf16, const void* A,
                                      const void* B, float* raw_out, int* status, void* stream) {
  using namespace atlas;
  if (!(M == 64 || M == 128) || N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16 || !A || !B ||
      !raw_out || !status)
    return ATLAS_ERR_INVALID_ARG;
  const int smem = 200 * 1024;  // generous: any descriptor misreading stays inside
  cudaFuncSetAttribute(k_selftest_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k_selftest_mma<<<1, 128, smem, (cudaStream_t)stream>>>(M, N, K, a_mn_major, b_mn_major, bf16, (const uint16_t*)A,
                                                         (const uint16_t*)B, raw_out, status);
  return cudaGetLastError() == cudaSuccess ? ATLAS_OK : ATLAS_ERR_CUDA;
}
