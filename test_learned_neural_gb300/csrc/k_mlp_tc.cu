// Fused chunked forward of the residual SiLU MLP memory without
// Newton-Schulz, on the tensor cores: memory width d = 64, hidden 256,
// chunks of C = 64 tokens, Omega window c = 1 (the Titans memory of
// titans-pytorch-mlx README, Eq. 12-14, with gradients taken at the chunk
// start, ATLAS summary Section 3.3, and post-update read-out, atlas-torch
// README "Known deviations from the paper's MAC").
//
// One cluster of 4 CTAs per (batch, head) unit; CTA q owns the hidden slice
// [64q, 64q + 64): W1[:, slice] (d x 64), W2[slice, :] (64 x d) and the same
// slices of S.  The kernel is persistent over the unit's chunks, so the fp32
// state never leaves the SM: it lives in TMEM lanes 16-31 of each 32-lane
// sub-partition, which the M = 64 accumulators (lanes 0-15) leave untouched.
// Per chunk, with row-vector tokens (X keys, R queries, V values; Kw = C
// window rows since c = 1):
//
//   Z  = X W1q                      A = SiLU(Z)
//   Yp = A W2q      -> summed over the 4 slices (DSMEM) -> dy = 2 gamma (X + sum - V)
//   dz = (dy W2q^T) * SiLU'(Z)
//   G1 = R X^T,  M1 = -Cw (.) G1
//   Zq = (B R) W1q + (D R) S1q + M1 dz              Aq = SiLU(Zq)
//   G2 = Aq A^T, M2 = -Cw (.) G2
//   Yq = (B Aq) W2q + (D Aq) S2q + M2 dy  -> summed over slices (DSMEM)
//   y  = R + sum_q Yq
//   S1q <- A_e S1q - X^T diag(cs_e) dz,  W1q <- B_e W1q + D_e S1q - X^T diag(cw_e) dz
//   S2q <- A_e S2q - A^T diag(cs_e) dy,  W2q <- B_e W2q + D_e S2q - A^T diag(cw_e) dy
//
// Cs, Cw, A_t, B_t, D_t are the momentum/decay coefficients of the chunk
// (scans over eta and 1 - alpha, see k_generic.cu); (B R) scales row t of R
// by B_t.  Every product is one
// tcgen05.mma chain (M = 64, fp16 operands, fp32 accumulation in TMEM); the
// operands live in shared memory in the core-matrix layout of tc.cuh, each
// written once and read K-major or MN-major as the product needs.
//
// Operand precision.  The memory's state decays over long sequences (to
// ~1e-8 on the 4096-token Titans workload), and every chunk's gradient is
// taken from operands rounded from that fp32 state, so relative rounding
// errors accumulate over the chunks.  The operands are fp16 (11 significant
// bits, 8x finer than bf16), each tile multiplied by a power of two that
// brings its values near 1, so fp16's exponent range never flushes a
// decayed state:
//   s1, s2   W1q/S1q and W2q/S2q and the activations derived from them
//            (A, Aq ~ s1; dz ~ s2), from the CTA-wide maximum of the state
//            each state update writes.  The scale is a function of that
//            state alone, so a call that starts from a chunk boundary's
//            state rounds exactly as one that runs through it;
//   sx[b]    the chunk's keys and queries (one scale per chunk buffer),
//            reduced from the prefetched registers a chunk ahead.
// Epilogues divide the fp32 accumulators by the product of their operands'
// scales; sums of terms with different scales use separate accumulators.
#include <cuda_fp16.h>

#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {
namespace {

constexpr int D = 64, HQ = 64, CS = 4, TOK = 64, NT = 256;
constexpr int TILE = 64 * 64 * 2;       // bf16 64x64 operand tile
constexpr int RGS = 1024;               // row-group stride of a 64-column tile
constexpr int RGS2 = 2048;              // of a 128-column tile
constexpr int F32T = 64 * 64 * 4;       // fp32 64x64 tile (swizzled rows)
constexpr long long kWait = 1ll << 31;
constexpr uint32_t kSliceBytes = (CS - 1) * 16 * 64 * 4;   // fp32 row quarters from the 3 peers
constexpr uint32_t kDyBytes = (CS - 1) * 16 * 64 * 2;      // fp16 dy rows from the 3 peers
// fixed powers of two on tiles whose values are O(1) but whose bounds grow
// with the gates: dy (2 gamma (k + Yp - v)), the state corrections' operands
// (cs, cw up to C times a step) and M2 (Cw times a Gram of activations)
constexpr float kDyS = 1.f / 64, kCorrS = 1.f / 16, kM2S = 1.f / 16;

// shared-memory map (bytes): bf16 operand tiles in the core-matrix layout.
// X, Cw and the gate vectors have two buffers by chunk parity: the next
// chunk's are filled while the current chunk waits on its cluster barriers.
constexpr int OW1 = 0, OS1 = OW1 + TILE, OW2 = OS1 + TILE, OS2 = OW2 + TILE;   // state operands
constexpr int OX0 = OS2 + TILE, OX1 = OX0 + TILE;                 // X by chunk parity
constexpr int OR_ = OX1 + TILE, OA = OR_ + TILE, ODY = OA + TILE, ODZ = ODY + TILE;
constexpr int OSP = ODZ + TILE;                                   // SiLU'(Z)
constexpr int ORB = OSP + TILE, ORD = ORB + TILE;                 // B_t r_t, D_t r_t; later B_t aq_t, D_t aq_t
constexpr int OM = ORD + TILE, OAQ = OM + TILE;                   // M1, later M2; SiLU(Zq)
constexpr int ODZS = OAQ + TILE, ODYS = ODZS + 2 * TILE;          // [cs.dz | cw.dz], [cs.dy | cw.dy]
constexpr int CWM = ODYS + 2 * TILE;                              // fp32 Cw[t][i], by chunk parity
constexpr int OBRN = ODZS, ODRN = ODZS + TILE;                    // next chunk's B_t r_t, D_t r_t (in ODZS)
constexpr int RED = CWM + 2 * F32T;                               // Yp slots, Yq slots (cluster-shared)
constexpr int VEC = RED + 2 * F32T;                               // gate vectors, by chunk parity
constexpr int VECN = 12 * 64;                                     // floats per gate-vector buffer
constexpr int SMEM_BYTES = VEC + 2 * VECN * 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory map exceeds a CTA's limit");

// vectors inside VEC
constexpr int V_TH = 0, V_ET = 64, V_BE = 128, V_GA = 192, V_AP = 256, V_BP = 320, V_DP = 384, V_CS = 448,
              V_CW = 512;
// B_t, D_t of the read-out: the post-update state's (= V_BP, V_DP) or, in
// pre-update mode, the previous token's (1, 0 for the chunk's first token)
constexpr int V_BR = 576, V_DR = 640;

// TMEM columns of the accumulators (lanes 0-15 of each sub-partition)
constexpr uint32_t C_Z = 0, C_YP = 64, C_ZQ = 192, C_ST1 = 256, C_ST2 = 384;
// G1 of the next chunk is formed after this chunk's W1 state update, in the
// columns of the consumed W1 corrections
constexpr uint32_t C_G1 = C_ST1;
constexpr uint32_t C_G2 = 64, C_YQ = 128;   // reuse after Yp, G1 are consumed
// TMEM columns of the fp32 state (lanes 16-31 of each sub-partition)
constexpr uint32_t S_W1 = 0, S_S1 = 64, S_W2 = 128, S_S2 = 192;

__device__ __forceinline__ int swz(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }
// slot rows of 64 fp32 (16 rows per sender) use the same chunk swizzle:
// 16 threads writing one column chunk of 16 rows spread over all banks
__device__ __forceinline__ int slot_idx(int sender, int r16, int c) { return sender * 1024 + swz(r16, c); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Bulk copy of `bytes` from this CTA's shared memory to a peer's (cluster
// address), completing `bytes` of the transaction count of the peer's
// mbarrier (cluster address); 16-byte aligned, multiple of 16 bytes.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the issuing thread's bulk copies have finished reading their sources
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// one arrival on *bar that also expects `bytes` more of transactions
__device__ __forceinline__ void mbar_arm_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(cta));
  return r;
}

// 8 consecutive values of one row, times `scale`, as fp16 into an operand tile
__device__ __forceinline__ void st_h8(uint8_t* tile, int rgs, int row, int col, const float* v, float scale) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(scale * v[2 * i], scale * v[2 * i + 1]);
  *reinterpret_cast<uint4*>(tile + tc::core_offset(row, col, rgs)) = *reinterpret_cast<uint4*>(h);
}
// the stored (scaled) values back as fp32
__device__ __forceinline__ void ld_h8(const uint8_t* tile, int rgs, int row, int col, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(tile + tc::core_offset(row, col, rgs));
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// 2^-e for m = f 2^e, f in [0.5, 1): the power of two that brings the
// largest magnitude m into [0.5, 1) (1 for m = 0 or not finite)
__device__ __forceinline__ float pow2_scale(float m) {
  if (!(m > 0.f) || !(m < 3.0e38f)) return 1.f;
  int e = (int)((__float_as_uint(m) >> 23) & 255u) - 126;   // normal m; subnormals give e = -126
  // kept within 2^+-60 so that products of three scales stay finite
  e = e < -60 ? -60 : (e > 60 ? 60 : e);
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// CTA-wide maxima in two halves around a barrier the kernel has anyway:
// each warp's maximum into slot[warp] (8 floats of shared memory) before
// it, the CTA's from the slot after it.  No other write to the slot comes
// before every thread has read it.
__device__ __forceinline__ void warp_max_to_slot(float v, float* slot) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) slot[threadIdx.x >> 5] = v;
}
__device__ __forceinline__ float slot_max(const float* slot) {
  float m = slot[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, slot[w]);
  return m;
}
__device__ __forceinline__ float cta_max(float v, float* slot) {
  warp_max_to_slot(v, slot);
  __syncthreads();
  return slot_max(slot);
}

// 64 x N (x K) product, fp16 operands, issued by one thread.  Each K step
// moves the operand start address by a fixed byte count, so the descriptors
// are built once and stepped by adding (bytes >> 4) to their address field.
__device__ __forceinline__ void mma64(uint32_t d, const uint8_t* a, int a_mn, int a_rgs, const uint8_t* b, int b_mn,
                                      int b_rgs, int N, int K, bool accumulate) {
  const uint32_t idesc = tc::idesc_f16(64, N, 0, a_mn, b_mn);
  uint64_t ad = a_mn ? tc::sdesc(tc::smem_u32(a), a_rgs, 128) : tc::sdesc(tc::smem_u32(a), 128, a_rgs);
  uint64_t bd = b_mn ? tc::sdesc(tc::smem_u32(b), b_rgs, 128) : tc::sdesc(tc::smem_u32(b), 128, b_rgs);
  const uint64_t astep = (uint64_t)((a_mn ? 2 * a_rgs : 256) >> 4), bstep = (uint64_t)((b_mn ? 2 * b_rgs : 256) >> 4);
  for (int ks = 0; ks < K / 16; ++ks) {
    tc::mma_f16(d, ad, bd, idesc, (ks > 0 || accumulate) ? 1u : 0u);
    ad += astep;
    bd += bstep;
  }
}

__device__ __forceinline__ void sync_smem_for_mma() {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// Raw inputs of one chunk held in registers: thread tid covers row
// r = tid % 64 of the k and q tiles, column groups g and g + 4 (g = tid / 64),
// 8 bf16 (or 8 fp32 as two float4) values each; for the cross-slice sums it
// also holds k, v, q of row 16 (cluster rank) + tid / 16, columns
// 4 (tid % 16) .. + 3; threads 0-63 hold token tid's gates.  Loaded one
// chunk ahead so global latency hides behind work.
struct Prefetch {
  uint4 k[2][2], q[2][2];   // [group][0: values 0-3 | 1: values 4-7] (fp32) or [group][0] (bf16)
  uint4 kd, vd, qd;         // 4 values: fp32, or bf16 in .x, .y
  float th, et, al, ga;
};

__device__ __forceinline__ uint4 ld_in4(const void* p, size_t i, int dt) {
  if (dt == ATLAS_BF16) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>((const uint16_t*)p + i));
    return make_uint4(a.x, a.y, 0u, 0u);
  }
  return __ldg(reinterpret_cast<const uint4*>((const float*)p + i));
}

__device__ __forceinline__ void unpack4(uint4 w, int dt, float* o) {
  if (dt == ATLAS_BF16) {
    o[0] = __uint_as_float(w.x << 16);
    o[1] = __uint_as_float(w.x & 0xFFFF0000u);
    o[2] = __uint_as_float(w.y << 16);
    o[3] = __uint_as_float(w.y & 0xFFFF0000u);
  } else {
    o[0] = __uint_as_float(w.x); o[1] = __uint_as_float(w.y); o[2] = __uint_as_float(w.z); o[3] = __uint_as_float(w.w);
  }
}

__device__ __forceinline__ void prefetch_chunk(Prefetch& p, int dt, const void* q, const void* k, const void* v,
                                               const float* theta, const float* eta, const float* alpha,
                                               const float* gamma, int u, int T, int Tst, int s, uint32_t qr) {
  const int tid = threadIdx.x, r = tid % 64, g = tid / 64;
  if (s >= T) return;
  for (int j = 0; j < 2; ++j) {
    const size_t base = ((size_t)u * Tst + s + r) * 64 + (g + 4 * j) * 8;
    if (dt == ATLAS_BF16) {
      p.k[j][0] = __ldg(reinterpret_cast<const uint4*>((const uint16_t*)k + base));
      p.q[j][0] = __ldg(reinterpret_cast<const uint4*>((const uint16_t*)q + base));
    } else {
      p.k[j][0] = __ldg(reinterpret_cast<const uint4*>((const float*)k + base));
      p.k[j][1] = __ldg(reinterpret_cast<const uint4*>((const float*)k + base + 4));
      p.q[j][0] = __ldg(reinterpret_cast<const uint4*>((const float*)q + base));
      p.q[j][1] = __ldg(reinterpret_cast<const uint4*>((const float*)q + base + 4));
    }
  }
  const size_t gd = ((size_t)u * Tst + s + 16 * qr + (tid >> 4)) * 64 + (tid & 15) * 4;
  p.kd = ld_in4(k, gd, dt);
  p.vd = ld_in4(v, gd, dt);
  p.qd = ld_in4(q, gd, dt);
  if (tid < 64) {
    const size_t gi = (size_t)u * Tst + s + tid;
    p.th = __ldg(theta + gi);
    p.et = __ldg(eta + gi);
    p.al = __ldg(alpha + gi);
    p.ga = gamma ? __ldg(gamma + gi) : 1.f;
  }
}

// logistic sigmoid through the hardware tanh: s(z) = (1 + tanh(z / 2)) / 2
__device__ __forceinline__ float sigmoid_fast(float z) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
  return fmaf(0.5f, t, 0.5f);
}

__device__ __forceinline__ void unpack8(const uint4* w, int dt, float* o) {
  if (dt == ATLAS_BF16) {
    const uint32_t a[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(a[i] << 16);
      o[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
    }
  } else {
    const uint4 x = w[0], y = w[1];
    o[0] = __uint_as_float(x.x); o[1] = __uint_as_float(x.y); o[2] = __uint_as_float(x.z); o[3] = __uint_as_float(x.w);
    o[4] = __uint_as_float(y.x); o[5] = __uint_as_float(y.y); o[6] = __uint_as_float(y.z); o[7] = __uint_as_float(y.w);
  }
}

// y rows [16q, 16q + 16) of the chunk at token s: r_t + the four slices'
// Yq from this CTA's slots (thread: row tid / 16, columns 4 (tid % 16) .. + 3)
__device__ __forceinline__ void y_rows(float* y, const float* slots, const float* qv, int u, int Tst, int s,
                                       uint32_t qr, bool& ovf) {
  const int tid = threadIdx.x, rl = tid >> 4, cc = (tid & 15) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int p = 0; p < CS; ++p) {
    const float4 t4 = *reinterpret_cast<const float4*>(slots + slot_idx(p, rl, cc));
    acc.x += t4.x; acc.y += t4.y; acc.z += t4.z; acc.w += t4.w;
  }
  const size_t gb = ((size_t)u * Tst + s + 16 * (int)qr + rl) * D + cc;
  const float4 o = make_float4(qv[0] + acc.x, qv[1] + acc.y, qv[2] + acc.z, qv[3] + acc.w);
  ovf |= !(isfinite(o.x) && isfinite(o.y) && isfinite(o.z) && isfinite(o.w));
  *reinterpret_cast<float4*>(y + gb) = o;
}

struct Ctx {
  uint64_t* bar;
  uint32_t phase;
  bool ok;
};

// commit the MMAs issued so far by thread 0 and wait for them (bounded)
__device__ __forceinline__ void commit_wait(Ctx& c) {
  if (threadIdx.x == 0 && c.ok) tc::mma_commit(c.bar);
  bool good = true;
  if (c.ok) good = tc::mbar_wait(c.bar, c.phase, kWait);
  c.phase ^= 1;
  const int failed = __syncthreads_or(!good);
  if (failed) c.ok = false;
  tc::fence_after_sync();
}

}  // namespace

__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(NT, 1)
    k_mlp_dual_tc(int T, int Tst, int dt, const void* __restrict__ q, const void* __restrict__ k, const void* __restrict__ v,
                  const float* __restrict__ theta, const float* __restrict__ eta, const float* __restrict__ alpha,
                  const float* __restrict__ gamma, const float* W0a, const float* W0b, const float* S0a,
                  const float* S0b, float* __restrict__ y, float* Woa, float* Wob, float* Soa, float* Sob,
                  int* status, int pre, int cwise) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint64_t xbar[3];   // arrivals of the peers' Yp slices, dy rows, Yq slices
  __shared__ uint32_t tbase;
  __shared__ float redm[3][8];   // CTA-wide maxima: W1/S1, W2/S2, the chunk's keys and queries
  float* vec = reinterpret_cast<float*>(sm + VEC);
  float* cwm = reinterpret_cast<float*>(sm + CWM);
  // An operand beyond fp16's range becomes inf in its fp32 accumulator, and
  // every accumulator feeds y or the state: a non-finite y or final state
  // marks the call (ATLAS_ERR_RANGE) instead of a check at every store.
  bool ovf = false;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int sp = warp & 3, half = warp >> 2;
  // M = 64 accumulators keep rows 16 sp .. 16 sp + 15 in lanes 0-15 of
  // sub-partition sp; the 16x32bx2 load gives thread `lane` row
  // 16 sp + lane % 16 and 16 columns starting at cb (all 32 lanes busy).
  // The state uses the same rows in lanes 16-31.
  const int row = 16 * sp + (lane & 15);
  const int cb = 32 * half + 16 * (lane >> 4);
  const uint32_t lb = ((uint32_t)(32 * sp) << 16) + 32 * half;
  const uint32_t ls = ((uint32_t)(32 * sp + 16) << 16) + 32 * half;
  const uint32_t qr = cluster_rank();
  const int u = blockIdx.x / CS;
  const int H = 4 * HQ;

  // operand scales: W1q/S1q and W2q/S2q of the current chunk (s1c, s2c) and
  // of the tiles its state updates write (s1n, s2n); the keys and queries of
  // chunk buffer 0 and 1 (sx0, sx1) and of the prefetched chunk (sxp)
  float s1c = 1.f, s2c = 1.f, s1n = 1.f, s2n = 1.f, sx0 = 1.f, sx1 = 1.f, sxp = 1.f;
  if (warp == 0) tc::tmem_alloc(&tbase, 512);
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    for (int i = 0; i < 3; ++i) {
      tc::mbar_init(&xbar[i], 1);
      mbar_arm_tx(&xbar[i], i == 1 ? kDyBytes : kSliceBytes);   // phase 0 of each
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  cluster_sync();   // every CTA's exchange barriers are initialised and armed
  const uint32_t tb = tbase;

  // ---- state slices in: W1[:, 64q:64q+64] (d x 64), W2[64q:64q+64, :] (64 x d)
  {
    const size_t i1 = ((size_t)u * D + row) * H + 64 * qr + cb;
    const size_t i2 = ((size_t)u * H + 64 * qr + row) * D + cb;
    const float* src[4] = {W0a + i1, S0a + i1, W0b + i2, S0b + i2};
    const uint32_t col[4] = {S_W1, S_S1, S_W2, S_S2};
    const int op[4] = {OW1, OS1, OW2, OS2};
    float x[4][16], mx[2] = {0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(x[m] + i) = *reinterpret_cast<const float4*>(src[m] + i);
      tc::tmem_st16_x2(tb + ls + col[m], x[m]);
#pragma unroll
      for (int i = 0; i < 16; ++i) mx[m >> 1] = fmaxf(mx[m >> 1], fabsf(x[m][i]));
    }
    s1c = pow2_scale(cta_max(mx[0], redm[0]));
    s2c = pow2_scale(cta_max(mx[1], redm[1]));
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      st_h8(sm + op[m], RGS, row, cb, x[m], m < 2 ? s1c : s2c);
      st_h8(sm + op[m], RGS, row, cb + 8, x[m] + 8, m < 2 ? s1c : s2c);
    }
    tc::tmem_st_wait();
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  Ctx cx{&bar, 0u, true};
  Prefetch pf;
  prefetch_chunk(pf, dt, q, k, v, theta, eta, alpha, gamma, u, T, Tst, 0, qr);
  float qprev[4] = {0.f, 0.f, 0.f, 0.f};   // q of the previous chunk's rows, for its deferred y
  float xkd[4], vvd[4], qcur[4];            // this chunk's k, v, q rows of the cross-slice sums
  float xkn[4], vvn[4], qnx[4];             // the next chunk's
  const uint32_t red_local = tc::smem_u32(sm + RED);
  // an M = 64 accumulator's row quarters: the owner's own quarter into its
  // slot, the others into the staging blocks (ODZS, 4 KB per owner)
  // (the partial is sc * acc[col], plus sc2 * acc[col2] when sc2 != 0)
  auto stage_slices = [&](uint32_t col, int slot_off, float sc, uint32_t col2, float sc2) {
    float v16[16], w16[16];
    tc::tmem_ld16_x2(tb + lb + col, v16);
    if (sc2 != 0.f) tc::tmem_ld16_x2(tb + lb + col2, w16);
    tc::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v16[i] = sc * v16[i] + (sc2 != 0.f ? sc2 * w16[i] : 0.f);
    const int owner = row >> 4;
    // my own quarter: my slot [qr] (= [owner]); the others: staging block [owner]
    float* base = owner == (int)qr ? reinterpret_cast<float*>(sm + RED + slot_off)
                                   : reinterpret_cast<float*>(sm + ODZS);
#pragma unroll
    for (int i = 0; i < 16; i += 4)
      *reinterpret_cast<float4*>(base + slot_idx(owner, row & 15, cb + i)) =
          make_float4(v16[i], v16[i + 1], v16[i + 2], v16[i + 3]);
    tc::fence_smem_to_async();   // staging is the bulk copies' source
    __syncthreads();
  };
  // thread 0: the three staged quarters to their owners' slots [qr]
  auto send_slices = [&](int slot_off, int xb) {
    for (uint32_t p = 1; p < CS; ++p) {
      const uint32_t dst = (qr + p) % CS;
      const uint32_t src = tc::smem_u32(sm + ODZS) + dst * 4096;
      bulk_to_peer(mapa(red_local + slot_off + qr * 4096, dst), src, 4096, mapa(tc::smem_u32(&xbar[xb]), dst));
    }
    bulk_commit();
  };
  // thread 0 waits for phase `parity` of exchange barrier xb (bounded); the
  // CTA barrier then makes the arrived data visible to every thread
  auto xwait = [&](int xb, uint32_t parity) {
    bool good = true;
    if (tid == 0 && cx.ok) good = tc::mbar_wait(&xbar[xb], parity, kWait);
    if (__syncthreads_or(!good)) cx.ok = false;
  };
  auto vecb = [&](int b) { return vec + b * VECN; };
  auto cwmb = [&](int b) { return cwm + b * (F32T / 4); };

  // raw inputs of the chunk at token sn (held in pf) into buffer bn and
  // registers; then prefetch the chunk after it
  auto load_chunk = [&](int sn, int bn) {
    float* vb = vecb(bn);
    const int r = tid % 64, g = tid / 64;
    float xk[2][8], xq[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      unpack8(pf.k[j], dt, xk[j]);
      unpack8(pf.q[j], dt, xq[j]);
    }
    const float sc = sxp;   // reduced from these registers beforehand
    if (bn) sx1 = sc; else sx0 = sc;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      st_h8(sm + (bn ? OX1 : OX0), RGS, r, (g + 4 * j) * 8, xk[j], sc);
      st_h8(sm + OR_, RGS, r, (g + 4 * j) * 8, xq[j], sc);
    }
    if (tid < 64) {
      vb[V_TH + tid] = pf.th;
      vb[V_ET + tid] = pf.et;
      vb[V_BE + tid] = 1.f - pf.al;
      vb[V_GA + tid] = pf.ga;
    }
    unpack4(pf.kd, dt, xkn);
    unpack4(pf.vd, dt, vvn);
    unpack4(pf.qd, dt, qnx);
    prefetch_chunk(pf, dt, q, k, v, theta, eta, alpha, gamma, u, T, Tst, sn + TOK, qr);
  };

  // largest magnitude of the prefetched keys and queries held by this thread
  auto pf_max = [&]() {
    float xk[8], xq[8], m = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      unpack8(pf.k[j], dt, xk);
      unpack8(pf.q[j], dt, xq);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(xk[i]), fabsf(xq[i])));
    }
    return m;
  };

  // gate scans of buffer bn (window of token t is {t})
  auto scan_chunk = [&](int bn) {
    float* vb = vecb(bn);
    float* cwp = cwmb(bn);
    if (cwise) {
      // chunk-wise update rule (titans-pytorch store path): the memory
      // changes once, at the chunk's last token, by S_e = eta_bar S_bar -
      // sum_i theta_i g_i, W_e = (1 - alpha_bar) W_bar + S_e with the chunk's
      // mean gates; every earlier token reads W_bar, the last reads W_e
      // (post) or W_bar (pre)
      if (tid < 64) {
        const int i = tid;
        const float th = vb[V_TH + i];
        for (int t = 0; t < TOK; ++t) cwp[swz(t, i)] = (t == TOK - 1 && !pre) ? th : 0.f;
        vb[V_CS + i] = th;
        vb[V_CW + i] = th;
      } else if (tid == 64) {
        float se = 0.f, sb = 0.f;
        for (int t = 0; t < TOK; ++t) {
          se += vb[V_ET + t];
          sb += vb[V_BE + t];
        }
        const float eb = se / TOK, bb = sb / TOK;   // mean eta, mean (1 - alpha)
        for (int t = 0; t < TOK; ++t) {
          const bool last = t == TOK - 1;
          vb[V_AP + t] = last ? eb : 0.f;
          vb[V_BP + t] = last ? bb : 1.f;
          vb[V_DP + t] = last ? eb : 0.f;
          vb[V_BR + t] = last && !pre ? bb : 1.f;
          vb[V_DR + t] = last && !pre ? eb : 0.f;
        }
      }
      return;
    }
    if (tid < 64) {  // column i = tid of Cs / Cw
      const int i = tid;
      float cs = 0.f, cw = 0.f;
      for (int t0 = 0; t0 < TOK; t0 += 8) {
        float et[8], th[8], be[8];   // loads ahead of the stores (same shared array)
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          et[qq] = vb[V_ET + t0 + qq];
          th[qq] = vb[V_TH + t0 + qq];
          be[qq] = vb[V_BE + t0 + qq];
        }
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          const float cw_prev = cw;
          cs = et[qq] * cs + (t0 + qq == i ? th[qq] : 0.f);
          cw = be[qq] * cw + cs;
          cwp[swz(t0 + qq, i)] = pre ? cw_prev : cw;   // read-out weights of token t0 + qq
        }
      }
      vb[V_CS + i] = cs;
      vb[V_CW + i] = cw;
    } else if (tid == 64) {
      float Ap = 1.f, Bp = 1.f, Dp = 0.f;
      for (int t0 = 0; t0 < TOK; t0 += 8) {
        float et[8], be[8];
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          et[qq] = vb[V_ET + t0 + qq];
          be[qq] = vb[V_BE + t0 + qq];
        }
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          const float Bprev = Bp, Dprev = Dp;
          Ap *= et[qq];
          Bp *= be[qq];
          Dp = be[qq] * Dp + Ap;
          vb[V_AP + t0 + qq] = Ap;
          vb[V_BP + t0 + qq] = Bp;
          vb[V_DP + t0 + qq] = Dp;
          vb[V_BR + t0 + qq] = pre ? Bprev : Bp;
          vb[V_DR + t0 + qq] = pre ? Dprev : Dp;
        }
      }
    }
  };

  // (B R), (D R): the read-out's state terms of buffer bn's chunk, into the
  // two 64-column tiles at ODZS (free from the corrections product of the
  // current chunk until the Yq staging at its end)
  auto brdr = [&](int bn) {
    const float* vb = vecb(bn);
    const int r = tid % 64, g = tid / 64;
    const float ir = 1.f / (bn ? sx1 : sx0);   // R is stored times the chunk's input scale
    const float Bt = vb[V_BR + r] * ir, Dt = vb[V_DR + r] * ir;
    for (int j = 0; j < 2; ++j) {
      const int cc = (g + 4 * j) * 8;
      float x[8], b8[8], d8[8];
      ld_h8(sm + OR_, RGS, r, cc, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) { b8[i] = Bt * x[i]; d8[i] = Dt * x[i]; }
      st_h8(sm + OBRN, RGS, r, cc, b8, 1.f);
      st_h8(sm + ODRN, RGS, r, cc, d8, 1.f);
    }
  };

  // one state half-update: S <- A_e S - corr_S, W <- B_e W + D_e S - corr_W
  // (ic: 1 / the product of the corrections' operand scales; slot: the
  // CTA-wide maximum's scratch; s_new: the new state's operand scale)
  auto state_update = [&](const float* vb, uint32_t c_corr, uint32_t s_w, uint32_t s_s, int ow, int os, float ic,
                          float* slot, float& s_new) {
    const float Ae = vb[V_AP + 63], Be = vb[V_BP + 63], De = vb[V_DP + 63];
    float scr[16], wcr[16], so[16], wo[16];
    tc::tmem_ld16_x2(tb + lb + c_corr, scr);
    tc::tmem_ld16_x2(tb + lb + c_corr + 64, wcr);
    tc::tmem_ld16_x2(tb + ls + s_s, so);
    tc::tmem_ld16_x2(tb + ls + s_w, wo);
    tc::tmem_ld_wait();
    float sn[16], wn[16], mx = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      sn[i] = Ae * so[i] - ic * scr[i];
      wn[i] = Be * wo[i] + De * so[i] - ic * wcr[i];
      mx = fmaxf(mx, fmaxf(fabsf(sn[i]), fabsf(wn[i])));
    }
    tc::tmem_st16_x2(tb + ls + s_s, sn);
    tc::tmem_st16_x2(tb + ls + s_w, wn);
    const float sc = pow2_scale(cta_max(mx, slot));
    s_new = sc;
    st_h8(sm + ow, RGS, row, cb, wn, sc);
    st_h8(sm + ow, RGS, row, cb + 8, wn + 8, sc);
    st_h8(sm + os, RGS, row, cb, sn, sc);
    st_h8(sm + os, RGS, row, cb + 8, sn + 8, sc);
    tc::tmem_st_wait();
  };

  // ---- first chunk's inputs, gate scans, (B R), (D R) and Z = X W1q
  sxp = pow2_scale(cta_max(pf_max(), redm[2]));
  load_chunk(0, 0);
  __syncthreads();   // every thread has read redm[2]
  warp_max_to_slot(pf_max(), redm[2]);   // chunk 1's, read after the next barrier
#pragma unroll
  for (int i = 0; i < 4; ++i) { xkd[i] = xkn[i]; vvd[i] = vvn[i]; qcur[i] = qnx[i]; }
  __syncthreads();
  sxp = pow2_scale(slot_max(redm[2]));
  scan_chunk(0);
  __syncthreads();
  brdr(0);
  sync_smem_for_mma();
  if (tid == 0 && cx.ok) {
    mma64(tb + C_Z, sm + OX0, 0, RGS, sm + OW1, 1, RGS, 64, 64, false);
    mma64(tb + C_G1, sm + OR_, 0, RGS, sm + OX0, 0, RGS, 64, 64, false);
    mma64(tb + C_ZQ, sm + OBRN, 0, RGS, sm + OW1, 1, RGS, 64, 64, false);
    mma64(tb + C_ZQ, sm + ODRN, 0, RGS, sm + OS1, 1, RGS, 64, 64, true);
  }
  commit_wait(cx);

  // Software pipeline: a chunk starts with its X, R, gates, gate scans,
  // (B R), (D R) in shared memory and Z = X W1q issued; the next chunk's
  // are prepared inside this chunk's cluster-barrier waits and tail.
  for (int s = 0, n = 0; s < T; s += TOK, ++n) {
    const int b = n & 1;
    const bool has_next = s + TOK < T;
    const float* vb = vecb(b);
    const float* cwc = cwmb(b);
    const uint8_t* oxc = sm + (b ? OX1 : OX0);
    // ---------------------------------------------------------------- 1: G1, Zq state terms
    // Z, G1 and Zq's state terms were formed with the previous chunk's tail
    // (or before the loop) and waited for there
    {
      float z[16], g[16];
      tc::tmem_ld16_x2(tb + lb + C_Z, z);
      tc::tmem_ld16_x2(tb + lb + C_G1, g);
      tc::tmem_ld_wait();
      const float sxc = b ? sx1 : sx0;
      const float iz = 1.f / (sxc * s1c), ig = 1.f / (sxc * sxc);   // Z = (sx X)(s1 W1), G1 = (sx R)(sx X)^T
      float a[16], spv[16], m1[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        z[i] *= iz;
        g[i] *= ig;
        const float sg = sigmoid_fast(z[i]);
        a[i] = z[i] * sg;
        spv[i] = sg * (1.f + z[i] * (1.f - sg));
      }
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 c4 = *reinterpret_cast<const float4*>(cwc + swz(row, cb + i));
        m1[i] = -c4.x * g[i]; m1[i + 1] = -c4.y * g[i + 1]; m1[i + 2] = -c4.z * g[i + 2]; m1[i + 3] = -c4.w * g[i + 3];
      }
      st_h8(sm + OA, RGS, row, cb, a, s1c);          // A ~ W1: scale s1
      st_h8(sm + OA, RGS, row, cb + 8, a + 8, s1c);
      st_h8(sm + OSP, RGS, row, cb, spv, 1.f);
      st_h8(sm + OSP, RGS, row, cb + 8, spv + 8, 1.f);
      st_h8(sm + OM, RGS, row, cb, m1, 1.f);
      st_h8(sm + OM, RGS, row, cb + 8, m1 + 8, 1.f);
    }
    sync_smem_for_mma();
    // ---------------------------------------------------------------- 2: Yp = A W2q
    if (tid == 0 && cx.ok) mma64(tb + C_YP, sm + OA, 0, RGS, sm + OW2, 1, RGS, 64, 64, false);
    commit_wait(cx);
    // Cross-slice sums are reduce-scatters over DSMEM: CTA p owns rows
    // [16p, 16p + 16).  Every CTA stages the row quarters of its partial
    // (fp32, 4 KB each; ODZS is free until the dz step), bulk-copies each to
    // its owner's slot [sender] with a transaction on the owner's xbar, and
    // writes its own quarter straight into its slot.  RED holds the Yp
    // slots, RED + F32T the Yq slots.  A slot is rewritten only after its
    // owner has read it: the owner reads before sending the next dy rows,
    // which every sender needs before its next slice is formed.
    if (tid == 0) bulk_wait_read();   // the previous Yq copies have left ODZS
    __syncthreads();
    stage_slices(C_YP, 0, 1.f / (s1c * s2c), 0u, 0.f);   // Yp = (s1 A)(s2 W2)
    if (tid == 0 && cx.ok) send_slices(0, 0);
    // while the peers' slices travel: the next chunk's inputs (R and its
    // buffers are free: this chunk's G1, (B R), (D R) products are done)
    if (has_next) load_chunk(s + TOK, b ^ 1);
    xwait(0, n & 1);
    if (tid == 0 && cx.ok && has_next) mbar_arm_tx(&xbar[0], kSliceBytes);
    // dy = 2 gamma (X + sum Yp - V) for my 16 rows into my dy operand tile,
    // then bulk-copied (2 KB: rows 16q .. 16q + 15 are two row groups) into
    // every peer's; the previous chunk's Yq slots are summed here too
    if (s > 0) xwait(2, (n - 1) & 1);
    {
      const float* red = reinterpret_cast<const float*>(sm + RED);
      const int rl = tid >> 4, cc = (tid & 15) * 4, r = 16 * (int)qr + rl;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int p = 0; p < CS; ++p) {
        const float4 t4 = *reinterpret_cast<const float4*>(red + slot_idx(p, rl, cc));
        acc.x += t4.x; acc.y += t4.y; acc.z += t4.z; acc.w += t4.w;
      }
      const float g2 = 2.f * vb[V_GA + r] * kDyS;
      const float d0 = g2 * (xkd[0] + acc.x - vvd[0]), d1 = g2 * (xkd[1] + acc.y - vvd[1]);
      const float d2 = g2 * (xkd[2] + acc.z - vvd[2]), d3 = g2 * (xkd[3] + acc.w - vvd[3]);
      const __half2 h0 = __floats2half2_rn(d0, d1);
      const __half2 h1 = __floats2half2_rn(d2, d3);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&h0);
      pk.y = *reinterpret_cast<const uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(sm + ODY + tc::core_offset(r, cc, RGS)) = pk;
      if (s > 0) y_rows(y, reinterpret_cast<const float*>(sm + RED + F32T), qprev, u, Tst, s - TOK, qr, ovf);
    }
    tc::fence_smem_to_async();   // the dy rows are the bulk copies' source
    __syncthreads();
    if (tid == 0) {
      // Yq slots read (the y rows above): the next Yq slices may come
      if (s > 0 && cx.ok) mbar_arm_tx(&xbar[2], kSliceBytes);
      if (cx.ok) {
        const uint32_t src = tc::smem_u32(sm + ODY + 2 * (int)qr * RGS);
        for (uint32_t p = 1; p < CS; ++p) {
          const uint32_t dst = (qr + p) % CS;
          bulk_to_peer(mapa(src, dst), src, 2 * RGS, mapa(tc::smem_u32(&xbar[1]), dst));
        }
        bulk_commit();
      }
    }
    // while the peers' dy rows travel: the next chunk's gate scans
    if (has_next) scan_chunk(b ^ 1);
    xwait(1, n & 1);
    if (tid == 0 && cx.ok && has_next) mbar_arm_tx(&xbar[1], kDyBytes);
    sync_smem_for_mma();
    // ---------------------------------------------------------------- 3: dz' = dy W2q^T
    if (tid == 0 && cx.ok) mma64(tb + C_Z, sm + ODY, 0, RGS, sm + OW2, 0, RGS, 64, 64, false);
    // state operand diag(cs | cw) dy from the broadcast dy tile (overlaps the product)
    {
      const int r = tid % 64, g = tid / 64;
      const float csr = kCorrS * vb[V_CS + r], cwr = kCorrS * vb[V_CW + r];
      for (int j = 0; j < 2; ++j) {
        const int cc = (g + 4 * j) * 8;
        float dy[8], t0[8], t1[8];
        ld_h8(sm + ODY, RGS, r, cc, dy);
#pragma unroll
        for (int i = 0; i < 8; ++i) { t0[i] = csr * dy[i]; t1[i] = cwr * dy[i]; }
        st_h8(sm + ODYS, RGS2, r, cc, t0, 1.f);
        st_h8(sm + ODYS, RGS2, r, 64 + cc, t1, 1.f);
      }
    }
    if (tid == 0) bulk_wait_read();   // the Yp copies have left ODZS (rewritten next)
    // the chunk after next (prefetched at stage 2): its input scale, reduced
    // at the barrier of the wait below
    if (has_next) warp_max_to_slot(pf_max(), redm[2]);
    commit_wait(cx);
    if (has_next) sxp = pow2_scale(slot_max(redm[2]));
    {
      float t[16], spv[16];
      tc::tmem_ld16_x2(tb + lb + C_Z, t);
      ld_h8(sm + OSP, RGS, row, cb, spv);
      ld_h8(sm + OSP, RGS, row, cb + 8, spv + 8);
      tc::tmem_ld_wait();
      const float csr = kCorrS * vb[V_CS + row], cwr = kCorrS * vb[V_CW + row];
      float t0[16], t1[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        t[i] *= spv[i];
        t0[i] = csr * t[i];
        t1[i] = cwr * t[i];
      }
      // t = dz' SiLU'(Z) = kDyS s2 dz (dy's fixed scale, W2's s2)
      st_h8(sm + ODZ, RGS, row, cb, t, 1.f);
      st_h8(sm + ODZ, RGS, row, cb + 8, t + 8, 1.f);
      st_h8(sm + ODZS, RGS2, row, cb, t0, 1.f);   // kCorrS is in csr, cwr
      st_h8(sm + ODZS, RGS2, row, cb + 8, t0 + 8, 1.f);
      st_h8(sm + ODZS, RGS2, row, 64 + cb, t1, 1.f);
      st_h8(sm + ODZS, RGS2, row, 64 + cb + 8, t1 + 8, 1.f);
    }
    sync_smem_for_mma();
    // ---------------------------------------------------------------- 4: Zq += M1 dz; state corrections
    if (tid == 0 && cx.ok) {
      // M1 dz into the Z columns (free: this chunk's Z and dz' are consumed);
      // its operands carry other scales than Zq's state terms
      mma64(tb + C_Z, sm + OM, 0, RGS, sm + ODZ, 1, RGS, 64, 64, false);
      mma64(tb + C_ST1, oxc, 1, RGS, sm + ODZS, 1, RGS2, 128, 64, false);    // X^T [cs dz | cw dz]
      mma64(tb + C_ST2, sm + OA, 1, RGS, sm + ODYS, 1, RGS2, 128, 64, false);   // A^T [cs dy | cw dy]
    }
    commit_wait(cx);
    {
      const float Bt = vb[V_BR + row], Dt = vb[V_DR + row];
      float zq[16], zm[16];
      tc::tmem_ld16_x2(tb + lb + C_ZQ, zq);
      tc::tmem_ld16_x2(tb + lb + C_Z, zm);
      tc::tmem_ld_wait();
      // state terms (B R)(s1 W1) + (D R)(s1 S1); M1 (kDyS s2 dz)
      const float iq = 1.f / s1c, im = 1.f / (kDyS * s2c);
      float aq[16], ab[16], ad[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        zq[i] = iq * zq[i] + im * zm[i];
        aq[i] = s1c * zq[i] * sigmoid_fast(zq[i]);   // Aq ~ W1: scale s1
        ab[i] = Bt * aq[i];
        ad[i] = Dt * aq[i];
      }
      st_h8(sm + OAQ, RGS, row, cb, aq, 1.f);
      st_h8(sm + OAQ, RGS, row, cb + 8, aq + 8, 1.f);
      st_h8(sm + ORB, RGS, row, cb, ab, 1.f);
      st_h8(sm + ORB, RGS, row, cb + 8, ab + 8, 1.f);
      st_h8(sm + ORD, RGS, row, cb, ad, 1.f);
      st_h8(sm + ORD, RGS, row, cb + 8, ad + 8, 1.f);
    }
    // W1, S1 are no longer read by this chunk's products.  Corrections:
    // (sx X)^T (kCorrS kDyS s2 [cs dz | cw dz])
    {
      const float sxc = b ? sx1 : sx0;
      state_update(vb, C_ST1, S_W1, S_S1, OW1, OS1, 1.f / (sxc * s2c * kCorrS * kDyS), redm[0], s1n);
    }
    // the corrections product has read ODZS: the next chunk's (B R), (D R)
    if (has_next) brdr(b ^ 1);
    sync_smem_for_mma();
    // ---------------------------------------------------------------- 5: G2, Yq state terms
    // and the next chunk's Z = X' W1q (W1 is final for this chunk)
    if (tid == 0 && cx.ok) {
      mma64(tb + C_G2, sm + OAQ, 0, RGS, sm + OA, 0, RGS, 64, 64, false);
      mma64(tb + C_YQ, sm + ORB, 0, RGS, sm + OW2, 1, RGS, 64, 64, false);
      mma64(tb + C_YQ, sm + ORD, 0, RGS, sm + OS2, 1, RGS, 64, 64, true);
      if (has_next) {
        // the next chunk's first products: W1, S1 are final for this chunk
        const uint8_t* oxn = sm + (b ? OX0 : OX1);
        mma64(tb + C_Z, oxn, 0, RGS, sm + OW1, 1, RGS, 64, 64, false);
        mma64(tb + C_G1, sm + OR_, 0, RGS, oxn, 0, RGS, 64, 64, false);
        mma64(tb + C_ZQ, sm + OBRN, 0, RGS, sm + OW1, 1, RGS, 64, 64, false);
        mma64(tb + C_ZQ, sm + ODRN, 0, RGS, sm + OS1, 1, RGS, 64, 64, true);
      }
    }
    commit_wait(cx);
    {
      float g[16], m2[16];
      tc::tmem_ld16_x2(tb + lb + C_G2, g);
      tc::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 c4 = *reinterpret_cast<const float4*>(cwc + swz(row, cb + i));
        m2[i] = -c4.x * g[i]; m2[i + 1] = -c4.y * g[i + 1]; m2[i + 2] = -c4.z * g[i + 2]; m2[i + 3] = -c4.w * g[i + 3];
      }
      // G2 = (s1 Aq)(s1 A)^T: M2 stays in that scale, times kM2S
      st_h8(sm + OM, RGS, row, cb, m2, kM2S);
      st_h8(sm + OM, RGS, row, cb + 8, m2 + 8, kM2S);
    }
    sync_smem_for_mma();
    // ---------------------------------------------------------------- 6: Yq += M2 dy
    // M2 dy into the G2 columns (consumed above): other scales than Yq's state terms
    if (tid == 0 && cx.ok) mma64(tb + C_G2, sm + OM, 0, RGS, sm + ODY, 1, RGS, 64, 64, false);
    // W2, S2 are no longer read by this chunk's products (overlaps the last
    // one).  Corrections: (s1 A)^T (kCorrS kDyS [cs dy | cw dy])
    state_update(vb, C_ST2, S_W2, S_S2, OW2, OS2, 1.f / (s1c * kCorrS * kDyS), redm[1], s2n);
    commit_wait(cx);
    // Yq = (s1 B Aq)(s2 W2) + (s1 D Aq)(s2 S2) + (kM2S s1^2 M2)(kDyS dy)
    stage_slices(C_YQ, F32T, 1.f / (s1c * s2c), C_G2, 1.f / (kM2S * kDyS * s1c * s1c));
    if (tid == 0 && cx.ok) send_slices(F32T, 2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qprev[i] = qcur[i];
      xkd[i] = xkn[i];
      vvd[i] = vvn[i];
      qcur[i] = qnx[i];
    }
    s1c = s1n;
    s2c = s2n;
    sync_smem_for_mma();
  }
  // the last chunk's y
  xwait(2, ((T / TOK) - 1) & 1);
  if (tid == 0) bulk_wait_all();   // every copy this CTA issued has landed
  __syncthreads();
  y_rows(y, reinterpret_cast<const float*>(sm + RED + F32T), qprev, u, Tst, T - TOK, qr, ovf);

  // ---- state slices out
  {
    const size_t i1 = ((size_t)u * D + row) * H + 64 * qr + cb;
    const size_t i2 = ((size_t)u * H + 64 * qr + row) * D + cb;
    float* dst[4] = {Woa + i1, Soa + i1, Wob + i2, Sob + i2};
    const uint32_t col[4] = {S_W1, S_S1, S_W2, S_S2};
    for (int m = 0; m < 4; ++m) {
      float x[16];
      tc::tmem_ld16_x2(tb + ls + col[m], x);
      tc::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4*>(dst[m] + i) = *reinterpret_cast<const float4*>(x + i);
#pragma unroll
      for (int i = 0; i < 16; ++i) ovf |= !isfinite(x[i]);
    }
  }
  if (!cx.ok && tid == 0) atomicExch(status, ATLAS_ERR_TIMEOUT);
  if (__syncthreads_or(ovf) && tid == 0) atomicCAS(status, 0, ATLAS_ERR_RANGE);
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();   // no CTA leaves while a peer may still read its shared memory
  if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

bool mlp_tc_supported(const Geom& g) {
  return g.depth == 2 && g.ns_iters == 0 && g.c == 1 && g.p == 1 && g.proj_dim == 0 && g.d_k == D &&
         g.d_v == D && g.hidden == 4 * HQ && g.C == TOK && g.n_prev == 0 && g.T % TOK == 0;
}

cudaError_t mlp_tc_launch(const Geom& g, const void* q, const void* k, const void* v, const float* theta,
                          const float* eta, const float* alpha, const float* gamma, const float* const* W0,
                          const float* const* S0, float* y, float* const* W_out, float* const* S_out, int* status,
                          cudaStream_t st, int Tst) {
  cudaError_t e = cudaFuncSetAttribute(k_mlp_dual_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  k_mlp_dual_tc<<<g.units * CS, NT, SMEM_BYTES, st>>>(g.T, Tst > 0 ? Tst : g.T, g.qkv_dtype, q, k, v, theta, eta,
                                                      alpha, gamma, W0[0],
                                                      W0[1], S0[0], S0[1], y, W_out[0], W_out[1], S_out[0],
                                                      S_out[1], status, g.readout == ATLAS_READOUT_PRE ? 1 : 0,
                                                      g.update == ATLAS_UPDATE_CHUNKWISE ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace atlas
