// Newton-Schulz orthogonalisation of the per-token momentum on the tensor
// cores (tcgen05, TMEM accumulators), for memories whose matrices have a
// short side of 64 (e.g. the 64 -> 256 -> 64 MLP memory).
//
// One task = (unit, token t of the chunk, weight matrix m).  For each task:
//   S_t  = A_t Sbar - Lx^T diag(Cs[t,:]) Rx        (momentum of token t, in
//          the orientation X whose short side comes first: r x n)
//   X_0  = S_t / (||S_t||_F + eps)
//   5x:  A = X X^T;  B' = a I + b A + c A^2;  X = B' X
//   U_t  = X_5  -> the token's slot of Ubuf (fp32)
// (atlas-torch README, "Atlas Extensions": Muon / Newton-Schulz; ATLAS
// summary, Section 5; titans-pytorch-mlx README, Eq. 14 for S_t.)
//
// Precision: the quintic map has slope 3.4445^5 ~ 485 at zero, so rounding
// in near-null directions is amplified; every product therefore runs as
// split bf16 (x = hi + lo, hi*hi' + hi*lo' + lo*hi', about 2^-16 relative)
// with fp32 accumulation in TMEM, and S_t, the norm and B' stay fp32.
//
// Shared-memory operands use the no-swizzle core-matrix layout of tc.cuh.
// X lives in one layout that is read as a K-major operand by X X^T and as an
// MN-major operand by B' X.
#include <cuda_bf16.h>

#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {

namespace {

constexpr int R = 64;     // short side of X
constexpr int NT = 256;   // threads per CTA: two warps per TMEM sub-partition
constexpr long long kWaitCycles = 1ll << 31;

struct NsSmem {
  // byte offsets inside dynamic shared memory
  int opr;        // factor operands, later X hi/lo
  int stg;        // fp32 staging of S (R x (n + 4)), later A / B' hi/lo
  int total;
};

__host__ __device__ inline NsSmem ns_smem_layout(int n, int Kp) {
  NsSmem s;
  const int lx = R * Kp * 2, rx = Kp * n * 2, xx = R * n * 2;
  int opr_bytes = 2 * lx + 2 * rx;
  if (opr_bytes < 2 * xx) opr_bytes = 2 * xx;
  const int stg_bytes = R * (n + 4) * 4;
  s.opr = 0;
  s.stg = (opr_bytes + 1023) & ~1023;
  s.total = s.stg + ((stg_bytes + 1023) & ~1023);
  return s;
}

__device__ inline void store_split16(uint8_t* hi, uint8_t* lo, uint32_t off, const float* v) {
  // 8 consecutive values of one row -> one 16-byte chunk in each array;
  // hi = bf16(x) and lo = bf16(x - hi), two values per conversion
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

// D (+)= A * B^T over K, split-bf16: hi*hi + hi*lo + lo*hi.
// A: K-major [M][K] (row-group stride aK); B: K-major [N][K] (b_mn = 0,
// row-group stride bK) or MN-major [K][N] (b_mn = 1, row-group stride bK).
__device__ inline void mma_x3(uint32_t d, const uint8_t* a_hi, const uint8_t* a_lo, int aK, const uint8_t* b_hi,
                              const uint8_t* b_lo, int bK, int b_mn, int M, int N, int K) {
  const uint32_t idesc = tc::idesc_f16(M, N, 1, 0, b_mn);
  const uint8_t* As[3] = {a_hi, a_hi, a_lo};
  const uint8_t* Bs[3] = {b_hi, b_lo, b_hi};
  for (int p = 0; p < 3; ++p)
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ad = tc::sdesc(tc::smem_u32(As[p]) + ks * 256, 128, aK);
      const uint64_t bd = b_mn ? tc::sdesc(tc::smem_u32(Bs[p]) + ks * 2 * bK, bK, 128)
                               : tc::sdesc(tc::smem_u32(Bs[p]) + ks * 256, 128, bK);
      tc::mma_f16(d, ad, bd, idesc, (p > 0 || ks > 0) ? 1u : 0u);
    }
}

// Every thread waits for the MMA group; the outcome is made uniform across
// the CTA (a timed-out wait anywhere aborts everyone).
__device__ inline bool wait_all(uint64_t* bar, uint32_t& phase) {
  const bool ok = tc::mbar_wait(bar, phase, kWaitCycles);
  phase ^= 1;
  const int failed = __syncthreads_or(!ok);
  tc::fence_after_sync();
  return failed == 0;
}

__device__ inline void sync_for_mma() {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

}  // namespace

// Persistent over tasks.  n = long side of X (multiple of 16, <= 256);
// Kp = window rows padded to a multiple of 16.
__global__ void __launch_bounds__(NT, 1) k_ns_tc64(Geom g, Chunk ch, Work w, int buf, size_t slot_stride, int n,
                                                    int Kp) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  __shared__ float red[NT / 32];
  const NsSmem L = ns_smem_layout(n, Kp);
  uint8_t* opr = sm + L.opr;
  float* stg = reinterpret_cast<float*>(sm + L.stg);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // M = 64 accumulators: rows 16 sp .. 16 sp + 15 sit in lanes 0-15 of
  // sub-partition sp.  With the 16x32bx2 load a warp reads 16 rows x 32
  // columns at once: thread `lane` gets row 16 sp + lane % 16 and columns
  // c + 16 (lane / 16) + [0, 16).  The two warps of a sub-partition take
  // alternate 32-column blocks (half = warp / 4).
  const int sp = warp & 3, half = warp >> 2;
  const int row = 16 * sp + (lane & 15);
  const int csub = 16 * (lane >> 4);
  const uint32_t lane_base = (uint32_t)(32 * sp) << 16;
  const int stg_ld = n + 4;

  if (warp == 0) tc::tmem_alloc(&tbase, 512);
  if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tA = tbase, tA2 = tbase + 64, tX = tbase + 128;
  uint32_t phase = 0;
  bool ok = true;

  // operand buffers inside opr / stg
  const int lxb = R * Kp * 2, rxb = Kp * n * 2, xb = R * n * 2, ab = R * R * 2;
  uint8_t* lx_hi = opr;
  uint8_t* lx_lo = opr + lxb;
  uint8_t* rx_hi = opr + 2 * lxb;
  uint8_t* rx_lo = opr + 2 * lxb + rxb;
  uint8_t* x_hi = opr;
  uint8_t* x_lo = opr + xb;
  uint8_t* a_hi = sm + L.stg;
  uint8_t* a_lo = sm + L.stg + ab;
  const int rgsKp = (Kp / 8) * 128, rgsN = (n / 8) * 128, rgsR = (R / 8) * 128;

  const int Ct = ch.e - ch.s;
  const int ntasks = g.units * g.nmat * Ct;
  for (int task = blockIdx.x; task < ntasks; task += gridDim.x) {
    const int r = task % Ct;
    const int m = (task / Ct) % g.nmat;
    const int u = task / (Ct * g.nmat);
    const int t = ch.s + r;
    const int rows = g.rows[m], cols = g.cols[m];
    const bool tall = rows > cols;
    // window factors: Lx gives the short-side index, Rx the long-side index
    const float* Lf;
    const float* Rf;
    int lstride, rstride;
    if (g.depth == 2 && m == 1) {        // W2 (h x d, tall): short side = d from dy, long = h from a
      Lf = w.DY + (size_t)u * g.Kw * g.d_v; lstride = g.d_v;
      Rf = w.Aact + (size_t)u * g.Kw * g.hidden; rstride = g.hidden;
    } else if (g.depth == 2) {           // W1 (d x h): short = d from x, long = h from dz
      Lf = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F; lstride = g.F;
      Rf = w.DZ + (size_t)u * g.Kw * g.hidden; rstride = g.hidden;
    } else {                             // depth 1 (F x d_v): orientation by shape
      const float* xf = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
      const float* dy = w.DY + (size_t)u * g.Kw * g.d_v;
      if (tall) { Lf = dy; lstride = g.d_v; Rf = xf; rstride = g.F; }
      else { Lf = xf; lstride = g.F; Rf = dy; rstride = g.d_v; }
    }
    const float* cs = w.Cs + ((size_t)u * g.C + r) * g.Kw;
    const float At = w.Ap[(size_t)u * g.C + r];
    const size_t nel = (size_t)rows * cols;
    const float* Sb = w.Sst[buf][m] + (size_t)u * nel;

    // (a) factors -> split-bf16 operands (zero rows beyond the window)
    for (int e = threadIdx.x; e < Kp * (R / 8); e += NT) {
      const int i = e / (R / 8), a0 = (e % (R / 8)) * 8;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = 0.f;
      if (i < ch.nw) {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = Lf[(size_t)i * lstride + a0 + q];
      }
      // Lx^T is the K-major A operand: row = short index a, k = window row i
      uint16_t h[8], l[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) tc::split_bf16(v[q], h[q], l[q]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t off = tc::core_offset(a0 + q, i, rgsKp);
        *reinterpret_cast<uint16_t*>(lx_hi + off) = h[q];
        *reinterpret_cast<uint16_t*>(lx_lo + off) = l[q];
      }
    }
    for (int e = threadIdx.x; e < Kp * (n / 8); e += NT) {
      const int i = e / (n / 8), b0 = (e % (n / 8)) * 8;
      float v[8];
      if (i < ch.nw) {
        const float c = cs[i];
        const float4 r0 = *reinterpret_cast<const float4*>(Rf + (size_t)i * rstride + b0);
        const float4 r1 = *reinterpret_cast<const float4*>(Rf + (size_t)i * rstride + b0 + 4);
        v[0] = c * r0.x; v[1] = c * r0.y; v[2] = c * r0.z; v[3] = c * r0.w;
        v[4] = c * r1.x; v[5] = c * r1.y; v[6] = c * r1.z; v[7] = c * r1.w;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
      // diag(cs) Rx is the MN-major B operand: k = window row i, n = long index b
      store_split16(rx_hi, rx_lo, tc::core_offset(i, b0, rgsN), v);
    }
    // (b) Sbar in the X orientation, fp32 staging
    if (!tall) {
      for (int e = threadIdx.x; e < R * n / 4; e += NT) {
        const int a = e / (n / 4), b = (e % (n / 4)) * 4;
        const float4 s4 = *reinterpret_cast<const float4*>(Sb + (size_t)a * n + b);
        *reinterpret_cast<float4*>(stg + a * stg_ld + b) = s4;
      }
    } else {
      for (int e = threadIdx.x; e < R * n; e += NT) {
        const int b = e / R, a = e % R;   // Sbar stored [b][a]
        stg[a * stg_ld + b] = Sb[e];
      }
    }
    sync_for_mma();
    // (c) D = Lx^T diag(cs) Rx   (M = 64, N = n, K = Kp)
    if (threadIdx.x == 0) {
      mma_x3(tX, lx_hi, lx_lo, rgsKp, rx_hi, rx_lo, rgsN, 1, R, n, Kp);
      tc::mma_commit(&bar);
    }
    if (!(ok = wait_all(&bar, phase))) break;
    // (d) S = A_t Sbar - D, in place in the staging; sum of squares
    float ss = 0.f;
    for (int c32 = 32 * half; c32 < n; c32 += 64) {
      float d[16];
      tc::tmem_ld16_x2(tX + lane_base + c32, d);
      tc::tmem_ld_wait();
      float* srow = stg + row * stg_ld + c32 + csub;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float s = At * srow[q] - d[q];
        srow[q] = s;
        ss += s * s;
      }
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    float tot = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < NT / 32; ++k2) tot += red[k2];
    const float scale = 1.f / (sqrtf(tot) + kNsEps);
    if (t == ch.e - 1) {   // chunk-end momentum, original orientation
      float* So = w.Sst[buf ^ 1][m] + (size_t)u * nel;
      for (int e = threadIdx.x; e < R * n; e += NT) {
        if (!tall) { const int a = e / n, b = e % n; So[e] = stg[a * stg_ld + b]; }
        else { const int b = e / R, a = e % R; So[e] = stg[a * stg_ld + b]; }
      }
    }
    // X_0 = S * scale -> split bf16 (opr region is free: the factor MMA is done)
    for (int c32 = 32 * half; c32 < n; c32 += 64)
      for (int h8 = 0; h8 < 16; h8 += 8) {
        float v[8];
        const int c = c32 + csub + h8;
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = stg[row * stg_ld + c + q] * scale;
        store_split16(x_hi, x_lo, tc::core_offset(row, c, rgsN), v);
      }
    sync_for_mma();

    float* slot = w.Ubuf + ((size_t)u * g.C + r) * slot_stride;
    for (int mm = 0; mm < m; ++mm) slot += (size_t)g.rows[mm] * g.cols[mm];
    for (int it = 0; it < g.ns_iters && ok; ++it) {
      // A = X X^T  (M = 64, N = 64, K = n; both operands K-major)
      if (threadIdx.x == 0) {
        mma_x3(tA, x_hi, x_lo, rgsN, x_hi, x_lo, rgsN, 0, R, R, n);
        tc::mma_commit(&bar);
      }
      if (!(ok = wait_all(&bar, phase))) break;
      {
        float v[16];
        const int c = 32 * half + csub;
        tc::tmem_ld16_x2(tA + lane_base + 32 * half, v);
        tc::tmem_ld_wait();
        store_split16(a_hi, a_lo, tc::core_offset(row, c, rgsR), v);
        store_split16(a_hi, a_lo, tc::core_offset(row, c + 8, rgsR), v + 8);
      }
      sync_for_mma();
      // A^2 (A symmetric: its rows serve as the K-major B operand)
      if (threadIdx.x == 0) {
        mma_x3(tA2, a_hi, a_lo, rgsR, a_hi, a_lo, rgsR, 0, R, R, R);
        tc::mma_commit(&bar);
      }
      if (!(ok = wait_all(&bar, phase))) break;
      {
        float va[16], v2[16], bp[16];
        const int c = 32 * half + csub;
        tc::tmem_ld16_x2(tA + lane_base + 32 * half, va);
        tc::tmem_ld16_x2(tA2 + lane_base + 32 * half, v2);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) bp[q] = kNsB * va[q] + kNsC * v2[q] + (row == c + q ? kNsA : 0.f);
        store_split16(a_hi, a_lo, tc::core_offset(row, c, rgsR), bp);
        store_split16(a_hi, a_lo, tc::core_offset(row, c + 8, rgsR), bp + 8);
      }
      sync_for_mma();
      // X = B' X  (M = 64, N = n, K = 64; X read as MN-major)
      if (threadIdx.x == 0) {
        mma_x3(tX, a_hi, a_lo, rgsR, x_hi, x_lo, rgsN, 1, R, n, R);
        tc::mma_commit(&bar);
      }
      if (!(ok = wait_all(&bar, phase))) break;
      const bool last = (it == g.ns_iters - 1);
      for (int c32 = 32 * half; c32 < n; c32 += 64) {
        float v[16];
        const int c = c32 + csub;
        tc::tmem_ld16_x2(tX + lane_base + c32, v);
        tc::tmem_ld_wait();
        if (last) {
          float4* o = reinterpret_cast<float4*>(slot + (size_t)row * n + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
          store_split16(x_hi, x_lo, tc::core_offset(row, c, rgsN), v);
          store_split16(x_hi, x_lo, tc::core_offset(row, c + 8, rgsN), v + 8);
        }
      }
      sync_for_mma();
    }
    if (!ok) break;
  }
  if (!ok && threadIdx.x == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

bool ns_tc_supported(const Geom& g) {
  if (g.ns_iters <= 0) return false;
  int n0 = -1;
  for (int m = 0; m < g.nmat; ++m) {
    const int s = g.rows[m] < g.cols[m] ? g.rows[m] : g.cols[m];
    const int l = g.rows[m] < g.cols[m] ? g.cols[m] : g.rows[m];
    if (s != R || l % 16 || l > 256) return false;
    if (n0 >= 0 && l != n0) return false;
    n0 = l;
  }
  const int Kp = (g.Kw + 15) / 16 * 16;
  if (Kp > 128) return false;
  return ns_smem_layout(n0, Kp).total <= 200 * 1024;
}

cudaError_t ns_tc_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, size_t slot_stride, int num_sms,
                         cudaStream_t st) {
  const int n = g.rows[0] < g.cols[0] ? g.cols[0] : g.rows[0];
  const int Kp = (g.Kw + 15) / 16 * 16;
  const int smem = ns_smem_layout(n, Kp).total;
  cudaFuncSetAttribute(k_ns_tc64, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int ntasks = g.units * g.nmat * (ch.e - ch.s);
  const int grid = ntasks < num_sms ? ntasks : num_sms;
  k_ns_tc64<<<grid, NT, smem, st>>>(g, ch, w, buf, slot_stride, n, Kp);
  return cudaGetLastError();
}

}  // namespace atlas
