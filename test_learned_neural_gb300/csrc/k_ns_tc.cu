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
// On this path the momentum state S of a matrix with rows > cols is kept
// transposed (the X orientation) for the whole call; ns_tc_state_in/out
// transpose it at the boundary.
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
  int rx;         // window factor on the long side, split bf16, unscaled (kept across a (unit, matrix)'s tokens)
  int lx;         // window factor on the short side, scaled by the token's coefficients
  int x;          // X hi, X lo (X lo directly after X hi: read together as one 128-row operand)
  int a;          // A, then B' (hi, lo; likewise adjacent)
  int qt;         // fp32 transpose buffer [64][65]
  int lf;         // window factor on the short side, fp32 [Kp][64], unscaled (kept like rx)
  int total;
};

__host__ __device__ inline NsSmem ns_smem_layout(int n, int Kp) {
  NsSmem s;
  s.rx = 0;
  s.lx = s.rx + 2 * Kp * n * 2;
  s.x = s.lx + 2 * R * Kp * 2;
  s.a = s.x + 2 * R * n * 2;
  s.qt = s.a + 2 * R * R * 2;
  s.lf = s.qt + R * (R + 1) * 4;
  s.total = s.lf + Kp * R * 4;
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
  // descriptors built once per product, stepped by (bytes >> 4) per K step
  const uint32_t idesc = tc::idesc_f16(M, N, 1, 0, b_mn);
  const uint8_t* As[3] = {a_hi, a_hi, a_lo};
  const uint8_t* Bs[3] = {b_hi, b_lo, b_hi};
  const uint64_t bstep = (uint64_t)((b_mn ? 2 * bK : 256) >> 4);
  for (int p = 0; p < 3; ++p) {
    uint64_t ad = tc::sdesc(tc::smem_u32(As[p]), 128, aK);
    uint64_t bd = b_mn ? tc::sdesc(tc::smem_u32(Bs[p]), bK, 128) : tc::sdesc(tc::smem_u32(Bs[p]), 128, bK);
    for (int ks = 0; ks < K / 16; ++ks) {
      tc::mma_f16(d, ad, bd, idesc, (p > 0 || ks > 0) ? 1u : 0u);
      ad += 256 >> 4;
      bd += bstep;
    }
  }
}

// D += A * B^T, as mma_x3 but accumulating onto D's previous contents
__device__ inline void mma_x3_acc(uint32_t d, const uint8_t* a_hi, const uint8_t* a_lo, int aK, const uint8_t* b_hi,
                                  const uint8_t* b_lo, int bK, int b_mn, int M, int N, int K) {
  const uint32_t idesc = tc::idesc_f16(M, N, 1, 0, b_mn);
  const uint8_t* As[3] = {a_hi, a_hi, a_lo};
  const uint8_t* Bs[3] = {b_hi, b_lo, b_hi};
  const uint64_t bstep = (uint64_t)((b_mn ? 2 * bK : 256) >> 4);
  for (int p = 0; p < 3; ++p) {
    uint64_t ad = tc::sdesc(tc::smem_u32(As[p]), 128, aK);
    uint64_t bd = b_mn ? tc::sdesc(tc::smem_u32(Bs[p]), bK, 128) : tc::sdesc(tc::smem_u32(Bs[p]), 128, bK);
    for (int ks = 0; ks < K / 16; ++ks) {
      tc::mma_f16(d, ad, bd, idesc, 1u);
      ad += 256 >> 4;
      bd += bstep;
    }
  }
}

// [P | Q] = Y_hi [Y_hi ; Y_lo]^T for a 64-row split-bf16 Y (K-major, Y_lo
// stored 8 row groups after Y_hi): one N = 128 chain instead of two N = 64.
__device__ inline void mma_hilo(uint32_t d, const uint8_t* y_hi, int rgs, int M, int K) {
  const uint32_t idesc = tc::idesc_f16(M, 2 * M, 1, 0, 0);
  uint64_t ad = tc::sdesc(tc::smem_u32(y_hi), 128, rgs);
  uint64_t bd = tc::sdesc(tc::smem_u32(y_hi), 128, rgs);
  for (int ks = 0; ks < K / 16; ++ks) {
    tc::mma_f16(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
    ad += 256 >> 4;
    bd += 256 >> 4;
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

// Persistent over tasks; CTA b takes a contiguous run of tasks ordered
// (unit, matrix, token), so the long-side window factor is split into
// bf16 hi/lo once per (unit, matrix) run and only the small short-side
// factor is rebuilt (scaled by the token's coefficients) per token.
// n = long side of X (multiple of 16, <= 256); Kp = window rows padded to a
// multiple of 16.
//
// X X^T and A^2 use the symmetry of the split: with Y = Y_hi + Y_lo,
// Y Y^T ~ P + Q + Q^T where [P | Q] = Y_hi [Y_hi ; Y_lo]^T is one N = 128
// product (Y_lo is stored right after Y_hi, so the pair is one 128-row
// operand); Q^T comes from a shared-memory transpose.
__global__ void __launch_bounds__(NT, 1) k_ns_tc64(Geom g, Chunk ch, Work w, int buf, size_t slot_stride, int n,
                                                    int Kp) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  __shared__ float red[NT / 32];
  const NsSmem L = ns_smem_layout(n, Kp);
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

  if (warp == 0) tc::tmem_alloc(&tbase, 512);
  if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tA = tbase, tA2 = tbase + 128, tX = tbase + 256;
  uint32_t phase = 0;
  bool ok = true;

  uint8_t* rx_hi = sm + L.rx;
  uint8_t* rx_lo = sm + L.rx + Kp * n * 2;
  uint8_t* lx_hi = sm + L.lx;
  uint8_t* lx_lo = sm + L.lx + R * Kp * 2;
  uint8_t* x_hi = sm + L.x;
  uint8_t* x_lo = sm + L.x + R * n * 2;
  uint8_t* a_hi = sm + L.a;
  uint8_t* a_lo = sm + L.a + R * R * 2;
  float* qt = reinterpret_cast<float*>(sm + L.qt);
  float* lfs = reinterpret_cast<float*>(sm + L.lf);
  // the chunk-start momentum S-bar of the current (unit, matrix), fp32, in
  // TMEM lanes 16-31 (the M = 64 accumulators use lanes 0-15), same row and
  // column layout as tX
  const uint32_t lane_sbar = (uint32_t)(32 * sp + 16) << 16;
  const int rgsKp = (Kp / 8) * 128, rgsN = (n / 8) * 128, rgsR = (R / 8) * 128;
  const int c = 32 * half + csub;           // this thread's 16 columns of a 64-wide accumulator

  const int rn = ns_first_row(g, ch), Cn = ch.e - ch.s - rn;   // tokens [rn, Ct) of the chunk
  const int ntasks = g.units * g.nmat * Cn;
  const int t_begin = (int)((long long)ntasks * blockIdx.x / gridDim.x);
  const int t_end = (int)((long long)ntasks * (blockIdx.x + 1) / gridDim.x);
  int loaded = -1;                          // (unit, matrix) whose long-side factor is resident
  for (int task = t_begin; task < t_end; ++task) {
    const int r = rn + task % Cn;
    const int m = (task / Cn) % g.nmat;
    const int u = task / (Cn * g.nmat);
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
    const float* Sb = w.Sst[buf][m] + (size_t)u * nel;   // X orientation [R][n]

    // (a) per (unit, matrix): long-side factor (MN-major B operand [Kp][n],
    // split bf16), short-side factor (fp32) and S-bar (TMEM)
    if (loaded != u * g.nmat + m) {
      loaded = u * g.nmat + m;
      for (int e = threadIdx.x; e < Kp * R; e += NT) {
        const int i = e / R, a = e % R;
        lfs[e] = i < ch.nw ? Lf[(size_t)i * lstride + a] : 0.f;
      }
      for (int c32 = 32 * half; c32 < n; c32 += 64) {
        const float* sb = Sb + (size_t)row * n + c32 + csub;
        float v[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) *reinterpret_cast<float4*>(v + 4 * q4) = *reinterpret_cast<const float4*>(sb + 4 * q4);
        tc::tmem_st16_x2(tA + lane_sbar + c32, v);
      }
      tc::tmem_st_wait();
      for (int e = threadIdx.x; e < Kp * (n / 8); e += NT) {
        const int i = e / (n / 8), b0 = (e % (n / 8)) * 8;
        float v[8];
        if (i < ch.nw) {
          const float4 r0 = *reinterpret_cast<const float4*>(Rf + (size_t)i * rstride + b0);
          const float4 r1 = *reinterpret_cast<const float4*>(Rf + (size_t)i * rstride + b0 + 4);
          v[0] = r0.x; v[1] = r0.y; v[2] = r0.z; v[3] = r0.w; v[4] = r1.x; v[5] = r1.y; v[6] = r1.z; v[7] = r1.w;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = 0.f;
        }
        store_split16(rx_hi, rx_lo, tc::core_offset(i, b0, rgsN), v);
      }
      __syncthreads();   // the fp32 short-side factor is read by other threads below
    }
    // short-side factor scaled by this token's coefficients: K-major A operand [R][Kp]
    for (int e = threadIdx.x; e < R * (Kp / 8); e += NT) {
      const int a = e % R, i0 = (e / R) * 8;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = (i0 + q < ch.nw) ? cs[i0 + q] * lfs[(i0 + q) * R + a] : 0.f;
      store_split16(lx_hi, lx_lo, tc::core_offset(a, i0, rgsKp), v);
    }
    sync_for_mma();
    // (b) D = (Lx diag cs)^T Rx   (M = 64, N = n, K = Kp)
    if (threadIdx.x == 0) {
      mma_x3(tX, lx_hi, lx_lo, rgsKp, rx_hi, rx_lo, rgsN, 1, R, n, Kp);
      tc::mma_commit(&bar);
    }
    if (!(ok = wait_all(&bar, phase))) break;
    // (c) S = A_t Sbar - D, straight into X in split bf16 (unscaled); sum of
    // squares; chunk-end S.  X_0 = s S with s = 1 / (||S||_F + eps) is
    // applied inside the first iteration (A = s^2 S S^T, X_1 = s B' S).
    float ss = 0.f;
    const bool last_tok = (t == ch.e - 1);
    float* So = w.Sst[buf ^ 1][m] + (size_t)u * nel;
    for (int c32 = 32 * half; c32 < n; c32 += 64) {
      float d[16], sv[16];
      tc::tmem_ld16_x2(tX + lane_base + c32, d);
      tc::tmem_ld16_x2(tA + lane_sbar + c32, sv);
      tc::tmem_ld_wait();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float* o = d + 4 * q4;
        const float* sbv = sv + 4 * q4;
        o[0] = At * sbv[0] - o[0]; o[1] = At * sbv[1] - o[1];
        o[2] = At * sbv[2] - o[2]; o[3] = At * sbv[3] - o[3];
        ss += o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
        if (last_tok) *reinterpret_cast<float4*>(So + (size_t)row * n + c32 + csub + 4 * q4) = make_float4(o[0], o[1], o[2], o[3]);
      }
      store_split16(x_hi, x_lo, tc::core_offset(row, c32 + csub, rgsN), d);
      store_split16(x_hi, x_lo, tc::core_offset(row, c32 + csub + 8, rgsN), d + 8);
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    sync_for_mma();
    float tot = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < NT / 32; ++k2) tot += red[k2];
    const float scale = 1.f / (sqrtf(tot) + kNsEps);

    float* slot = w.Ubuf + ((size_t)u * g.C + r) * slot_stride;
    for (int mm = 0; mm < m; ++mm) slot += (size_t)g.rows[mm] * g.cols[mm];
    for (int it = 0; it < g.ns_iters && ok; ++it) {
      // [P | Q] = X_hi [X_hi ; X_lo]^T   (M = 64, N = 128, K = n)
      if (threadIdx.x == 0) {
        mma_hilo(tA, x_hi, rgsN, R, n);
        tc::mma_commit(&bar);
      }
      if (!(ok = wait_all(&bar, phase))) break;
      float av[16];
      {
        float p[16], qv[16];
        tc::tmem_ld16_x2(tA + lane_base + 32 * half, p);
        tc::tmem_ld16_x2(tA + lane_base + 64 + 32 * half, qv);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) qt[row * (R + 1) + c + q] = qv[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 16; ++q) av[q] = p[q] + qv[q] + qt[(c + q) * (R + 1) + row];
        if (it == 0) {
#pragma unroll
          for (int q = 0; q < 16; ++q) av[q] *= scale * scale;
        }
        store_split16(a_hi, a_lo, tc::core_offset(row, c, rgsR), av);
        store_split16(a_hi, a_lo, tc::core_offset(row, c + 8, rgsR), av + 8);
      }
      sync_for_mma();
      // [P2 | Q2] = A_hi [A_hi ; A_lo]^T  (A symmetric: its rows are the K-major B operand)
      if (threadIdx.x == 0) {
        mma_hilo(tA2, a_hi, rgsR, R, R);
        tc::mma_commit(&bar);
      }
      if (!(ok = wait_all(&bar, phase))) break;
      {
        float p[16], qv[16], bp[16];
        tc::tmem_ld16_x2(tA2 + lane_base + 32 * half, p);
        tc::tmem_ld16_x2(tA2 + lane_base + 64 + 32 * half, qv);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) qt[row * (R + 1) + c + q] = qv[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float a2 = p[q] + qv[q] + qt[(c + q) * (R + 1) + row];
          bp[q] = kNsB * av[q] + kNsC * a2 + (row == c + q ? kNsA : 0.f);
        }
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
      // U rows go out through shared memory (row stride n + 4 floats over
      // the X and A buffers, free once B'X is done), one bulk copy per row
      float* ust = reinterpret_cast<float*>(sm + L.x);
      const int us = n + 4;
      for (int c32 = 32 * half; c32 < n; c32 += 64) {
        float v[16];
        const int cc = c32 + csub;
        tc::tmem_ld16_x2(tX + lane_base + c32, v);
        tc::tmem_ld_wait();
        if (it == 0) {
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] *= scale;   // X_1 = s B' S
        }
        if (last) {
          float4* o = reinterpret_cast<float4*>(ust + row * us + cc);
#pragma unroll
          for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
          store_split16(x_hi, x_lo, tc::core_offset(row, cc, rgsN), v);
          store_split16(x_hi, x_lo, tc::core_offset(row, cc + 8, rgsN), v + 8);
        }
      }
      if (last) {
        tc::fence_smem_to_async();
        __syncthreads();
        if (threadIdx.x < R) {
          const float* src = ust + threadIdx.x * us;
          float* dst = slot + (size_t)threadIdx.x * n;
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(tc::smem_u32(src)),
                       "r"(n * 4)
                       : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // the staging is rewritten by the next token
        }
      }
      sync_for_mma();
    }
    if (!ok) break;
  }
  if (threadIdx.x < R) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // the U rows
  if (!ok && threadIdx.x == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

// ============================================================ short side 128
// Matrices with a short side of 128 and a long side of 512 (the 128 -> 512
// -> 128 MLP memory).  X in split bf16 (256 KB) does not fit one SM, so a
// cluster of two CTAs shares each task: CTA p holds columns [256 p, 256 p +
// 256) of X.  X X^T = sum of the two halves' Gram matrices.  Each partial is
// symmetric, so a CTA sends the partner only its unique entries: block
// (0, 1) (16 KB fp32) and the two symmetric diagonal blocks' triangles
// packed into one 64 x 65 block (16.25 KB), one bulk DSMEM copy that
// completes on the partner's mbarrier (a copy between the two SMs moves
// about 19 bytes per cycle, so the bytes set the exchange's cost).  The
// receiver reads block (1, 0) as the transpose of block (0, 1) and the
// other triangles by symmetry.  A^2 and B' are formed redundantly by both;
// X <- B' X splits by columns with no exchange.
namespace {

constexpr int R2 = 128, NH = 256, NT2 = 256;
constexpr int OPR2 = 131072;                    // factors (120 KB) / X hi+lo (128 KB)
constexpr int AB2 = 65536;                      // A / B' hi+lo; receives the partner's partial
constexpr int STG2 = OPR2 + AB2;                // staging of this CTA's packed partial
constexpr int kQS = 65;                          // row stride of the packed diagonal blocks
// block (0, 1) [64][64] (16-byte chunks swizzled by xswz64), then Q
// [64][65]: row i holds P00[i][0..i] at columns 0..i and P11[i][i..63] at
// columns i+1..64 (65 = 1 mod 32: a row read and a column read of Q by 32
// consecutive rows both hit 32 banks)
constexpr uint32_t kPartBytes = 64 * 64 * 4 + 64 * kQS * 4;
constexpr int SMEM2 = STG2 + (int)kPartBytes;
// fp32 staging of the U rows: row stride 260 floats (1040 bytes = 16 mod
// 128, so the same 16-byte chunk of 8 consecutive rows hits 8 bank groups)
constexpr int kUS = 260;
static_assert(R2 * kUS * 4 <= STG2, "U staging fits the X and A/B' buffers");

__device__ __forceinline__ uint32_t cluster_rank2() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync2() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa2(uint32_t saddr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(cta));
  return r;
}
// bulk copy of local shared memory into the partner's, completing on the
// partner's mbarrier (cluster addresses for dst and mbar)
__device__ __forceinline__ void bulk_to_partner(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(src), "r"(bytes), "r"(mbar)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// bulk copy of local shared memory to global memory (both 16-byte aligned)
__device__ __forceinline__ void bulk_to_global(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read2() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all2() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void mbar_arm_tx2(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
// fp32 row-major exchange block with the 16-byte chunks of row r XOR-ed by
// r % 8: a warp touching one chunk of 32 consecutive rows hits every bank
// (unswizzled, rows 256 bytes apart all start in the same bank)
__device__ __forceinline__ int xswz64(int r, int c) { return r * 64 + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3)); }
// one arrival on the partner's mbarrier (cluster address)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

struct PairCtx {
  uint64_t* bar;
  uint32_t phase;
  bool ok;
};

// Bounded wait that never leaves the loop structure: after a timeout the
// CTA stops issuing and waiting, but keeps meeting its partner at every
// cluster barrier so neither can hang the other.
__device__ __forceinline__ void pair_commit_wait(PairCtx& c) {
  if (threadIdx.x == 0 && c.ok) tc::mma_commit(c.bar);
  bool good = true;
  if (c.ok) good = tc::mbar_wait(c.bar, c.phase, kWaitCycles);
  c.phase ^= 1;
  if (__syncthreads_or(!good)) c.ok = false;
  tc::fence_after_sync();
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT2, 1)
    k_ns_tc128(Geom g, Chunk ch, Work w, int buf, size_t slot_stride, int Kp, const float* __restrict__ theta,
               const float* __restrict__ eta) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  __shared__ float red[NT2 / 32];
  const uint32_t p = cluster_rank2();
  const int cl = blockIdx.x / 2, ncl = gridDim.x / 2;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int sp = warp & 3, half = warp >> 2;
  const int row = 32 * sp + lane;                   // M = 128: lane i of sub-partition sp holds row 32 sp + i
  const uint32_t lane_base = (uint32_t)(32 * sp) << 16;
  const int n = 2 * NH;                             // long side of X

  __shared__ uint64_t xdata, xfree;   // partner's partial arrived / partner ready to receive
  if (warp == 0) tc::tmem_alloc(&tbase, 512);
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init(&xdata, 1);
    tc::mbar_init(&xfree, 1);
    mbar_arm_tx2(&xdata, kPartBytes);   // exchange 0
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  cluster_sync2();   // both CTAs' exchange barriers are initialised
  // One arrival on the partner's xfree per exchange, as soon as this CTA's
  // A/B' buffer is free for it: after each token's momentum product (its
  // factors may reach into the buffer) and after every B'X product but a
  // token's last.
  const uint32_t xfree_peer = mapa2(tc::smem_u32(&xfree), p ^ 1u);
  // TMEM: the B'X product and, before it, A = X X^T and A^2 in its two
  // halves (each consumed before the next product writes there); the
  // running momentum of the current (unit, matrix) in the other 256 columns
  const uint32_t tX = tbase, tA = tbase, tA2 = tbase + 128, tS = tbase + 256;
  PairCtx cx{&bar, 0u, true};
  uint32_t xe = 0;   // exchanges so far (phase parity of xdata and xfree)
  float* stg = reinterpret_cast<float*>(sm + STG2);    // this CTA's packed partial
  float* recv = reinterpret_cast<float*>(sm + OPR2);   // the partner's (inside the A/B' buffer)

  const int lxb = R2 * Kp * 2, rxb = Kp * NH * 2;
  uint8_t* lx_hi = sm;
  uint8_t* lx_lo = sm + lxb;
  uint8_t* rx_hi = sm + 2 * lxb;
  uint8_t* rx_lo = sm + 2 * lxb + rxb;
  // the window update of one token: K = 16 rows (c <= 16)
  constexpr int KW = 16;
  const int lwb = R2 * KW * 2, rwb = KW * NH * 2;
  uint8_t* lw_hi = sm;
  uint8_t* lw_lo = sm + lwb;
  uint8_t* rw_hi = sm + 2 * lwb;
  uint8_t* rw_lo = sm + 2 * lwb + rwb;
  uint8_t* x_hi = sm;
  uint8_t* x_lo = sm + R2 * NH * 2;
  uint8_t* a_hi = sm + OPR2;
  uint8_t* a_lo = sm + OPR2 + R2 * R2 * 2;
  const int rgsKp = (Kp / 8) * 128, rgsN = (NH / 8) * 128, rgsR = (R2 / 8) * 128, rgsKW = (KW / 8) * 128;

  const int rn = ns_first_row(g, ch), Cn = ch.e - ch.s - rn;   // tokens [rn, Ct) of the chunk
  const int ntasks = g.units * g.nmat * Cn;
  // each CTA pair takes a contiguous run of tasks ordered (unit, matrix,
  // token), so within a run the momentum steps from one token to the next
  const int t_begin = (int)((long long)ntasks * cl / ncl), t_end = (int)((long long)ntasks * (cl + 1) / ncl);
  // momentum held in tS: S_t = lam * Shat for (unit, matrix) cur_um at token cur_r
  int cur_um = -1, cur_r = -1;
  float lam = 1.f;
  for (int task = t_begin; task < t_end; ++task) {
    const int r = rn + task % Cn;
    const int m = (task / Cn) % g.nmat;
    const int u = task / (Cn * g.nmat);
    const int t = ch.s + r;
    const int rows = g.rows[m], cols = g.cols[m];
    const bool tall = rows > cols;
    const float* Lf;
    const float* Rf;
    int lstride, rstride;
    if (g.depth == 2 && m == 1) {
      Lf = w.DY + (size_t)u * g.Kw * g.d_v; lstride = g.d_v;
      Rf = w.Aact + (size_t)u * g.Kw * g.hidden; rstride = g.hidden;
    } else if (g.depth == 2) {
      Lf = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F; lstride = g.F;
      Rf = w.DZ + (size_t)u * g.Kw * g.hidden; rstride = g.hidden;
    } else {
      const float* xf = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
      const float* dy = w.DY + (size_t)u * g.Kw * g.d_v;
      if (tall) { Lf = dy; lstride = g.d_v; Rf = xf; rstride = g.F; }
      else { Lf = xf; lstride = g.F; Rf = dy; rstride = g.d_v; }
    }
    const size_t nel = (size_t)rows * cols;
    const float* Sb = w.Sst[buf][m] + (size_t)u * nel;   // X orientation [128][512]
    // the token's momentum steps from the previous one held in TMEM
    // (titans-pytorch-mlx README, Eq. 14): S_t = eta_t S_{t-1} - theta_t g_t
    // with g_t the sum of the window rows' gradients (gamma folded in)
    const bool incr = cur_um == u * g.nmat + m && r == cur_r + 1 && g.update != ATLAS_UPDATE_CHUNKWISE &&
                      g.c <= KW;
    if (!incr) {
      // (a) full: factors Lx^T (K-major [128][Kp]) and this CTA's columns of
      // diag(cs) Rx, then S_t = A_t Sbar - Lx^T diag(cs) Rx into tS
      const float* cs = w.Cs + ((size_t)u * g.C + r) * g.Kw;
      const float At = w.Ap[(size_t)u * g.C + r];
      for (int e = threadIdx.x; e < R2 * (Kp / 8); e += NT2) {
        const int a = e % R2, i0 = (e / R2) * 8;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = (i0 + q < ch.nw) ? Lf[(size_t)(i0 + q) * lstride + a] : 0.f;
        store_split16(lx_hi, lx_lo, tc::core_offset(a, i0, rgsKp), v);
      }
      for (int e = threadIdx.x; e < Kp * (NH / 8); e += NT2) {
        const int i = e / (NH / 8), b0 = (e % (NH / 8)) * 8;
        float v[8];
        if (i < ch.nw) {
          const float c = cs[i];
          const float* src = Rf + (size_t)i * rstride + p * NH + b0;
          const float4 r0 = *reinterpret_cast<const float4*>(src);
          const float4 r1 = *reinterpret_cast<const float4*>(src + 4);
          v[0] = c * r0.x; v[1] = c * r0.y; v[2] = c * r0.z; v[3] = c * r0.w;
          v[4] = c * r1.x; v[5] = c * r1.y; v[6] = c * r1.z; v[7] = c * r1.w;
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = 0.f;
        }
        store_split16(rx_hi, rx_lo, tc::core_offset(i, b0, rgsN), v);
      }
      sync_for_mma();
      if (threadIdx.x == 0 && cx.ok) mma_x3(tX, lx_hi, lx_lo, rgsKp, rx_hi, rx_lo, rgsN, 1, R2, NH, Kp);
      pair_commit_wait(cx);
      for (int c32 = 32 * half; c32 < NH; c32 += 64) {
        float d[32];
        tc::tmem_ld16(tX + lane_base + c32, d);
        tc::tmem_ld16(tX + lane_base + c32 + 16, d + 16);
        const float* sb = Sb + (size_t)row * n + p * NH + c32;
        float4 s4[8];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) s4[q4] = *reinterpret_cast<const float4*>(sb + 4 * q4);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          float* o = d + 4 * q4;
          o[0] = At * s4[q4].x - o[0]; o[1] = At * s4[q4].y - o[1];
          o[2] = At * s4[q4].z - o[2]; o[3] = At * s4[q4].w - o[3];
        }
        tc::tmem_st16(tS + lane_base + c32, d);
        tc::tmem_st16(tS + lane_base + c32 + 16, d + 16);
      }
      tc::tmem_st_wait();
      lam = 1.f;
    } else {
      // (a') incremental: lam_t = lam_{t-1} eta_t; Shat_t = Shat_{t-1} -
      // (theta_t / lam_t) sum_{i in window(t)} Lf_i^T Rf_i (window rows
      // w0 .. t - lo of the chunk's factors; K = 16 padded with zeros)
      const size_t gi = (size_t)u * g.T + t;
      const int wt = t - ch.lo;                               // window row of token t
      const int w0 = (t - g.c + 1 > ch.lo ? t - g.c + 1 : ch.lo) - ch.lo;
      // every global read of this step is issued first (one round trip):
      // eta_t, theta_t, this thread's 8 short-side values (column a, rows
      // i0 .. i0 + 7 of the window) and 2 x 8 long-side values
      static_assert(R2 * (KW / 8) == NT2 && KW * (NH / 8) == 2 * NT2, "one / two staging items per thread");
      const float eta_t = __ldg(eta + gi), theta_t = __ldg(theta + gi);
      const int la = threadIdx.x % R2, li0 = (threadIdx.x / R2) * 8;
      float lv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = w0 + li0 + q;
        lv[q] = (i <= wt) ? Lf[(size_t)i * lstride + la] : 0.f;
      }
      float4 rv[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = threadIdx.x + h * NT2, i = w0 + e / (NH / 8), b0 = (e % (NH / 8)) * 8;
        if (i <= wt) {
          const float* src = Rf + (size_t)i * rstride + p * NH + b0;
          rv[2 * h] = *reinterpret_cast<const float4*>(src);
          rv[2 * h + 1] = *reinterpret_cast<const float4*>(src + 4);
        } else {
          rv[2 * h] = rv[2 * h + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      lam *= eta_t;
      if (!(lam > 1e-6f)) {
        // renormalise: Shat <- lam Shat, lam <- 1 (keeps theta / lam finite)
        for (int c32 = 32 * half; c32 < NH; c32 += 64) {
          float d[32];
          tc::tmem_ld16(tS + lane_base + c32, d);
          tc::tmem_ld16(tS + lane_base + c32 + 16, d + 16);
          tc::tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q) d[q] *= lam;
          tc::tmem_st16(tS + lane_base + c32, d);
          tc::tmem_st16(tS + lane_base + c32 + 16, d + 16);
        }
        tc::tmem_st_wait();
        lam = 1.f;
      }
      const float coef = -theta_t / lam;
#pragma unroll
      for (int q = 0; q < 8; ++q) lv[q] *= coef;
      store_split16(lw_hi, lw_lo, tc::core_offset(la, li0, rgsKW), lv);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = threadIdx.x + h * NT2, k = e / (NH / 8), b0 = (e % (NH / 8)) * 8;
        const float v[8] = {rv[2 * h].x, rv[2 * h].y, rv[2 * h].z, rv[2 * h].w,
                            rv[2 * h + 1].x, rv[2 * h + 1].y, rv[2 * h + 1].z, rv[2 * h + 1].w};
        store_split16(rw_hi, rw_lo, tc::core_offset(k, b0, rgsN), v);
      }
      sync_for_mma();
      if (threadIdx.x == 0 && cx.ok) mma_x3_acc(tS, lw_hi, lw_lo, rgsKW, rw_hi, rw_lo, rgsN, 1, R2, NH, KW);
      pair_commit_wait(cx);
    }
    // the momentum product is done: the partner may send this token's first exchange
    if (threadIdx.x == 0 && cx.ok) mbar_arrive_remote(xfree_peer);
    cur_um = u * g.nmat + m;
    cur_r = r;
    // (c) Shat itself, unscaled, in split bf16 as this CTA's half of X, and
    // the chunk-end S = lam Shat.  X_0 = s Shat with s = lam / (lam
    // ||Shat||_F + eps); ||Shat||^2 is the trace of Shat Shat^T, i.e. of the
    // first iteration's A before scaling, so s is applied there (A = s^2
    // Shat Shat^T, X_1 = s B' Shat) and needs no pass or exchange of its own.
    const bool last_tok = (t == ch.e - 1);
    float* So = w.Sst[buf ^ 1][m] + (size_t)u * nel;
    for (int c32 = 32 * half; c32 < NH; c32 += 64) {
      float d[32];
      tc::tmem_ld16(tS + lane_base + c32, d);
      tc::tmem_ld16(tS + lane_base + c32 + 16, d + 16);
      tc::tmem_ld_wait();
      if (last_tok) {
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4*>(So + (size_t)row * n + p * NH + c32 + 4 * q4) =
              make_float4(lam * d[4 * q4], lam * d[4 * q4 + 1], lam * d[4 * q4 + 2], lam * d[4 * q4 + 3]);
      }
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) store_split16(x_hi, x_lo, tc::core_offset(row, c32 + 8 * q8, rgsN), d + 8 * q8);
    }
    sync_for_mma();
    float scale = 1.f;   // s, from the first iteration's A
    float* slot = w.Ubuf + ((size_t)u * g.C + r) * slot_stride;
    for (int mm = 0; mm < m; ++mm) slot += (size_t)g.rows[mm] * g.cols[mm];
    for (int it = 0; it < g.ns_iters; ++it) {
      // partial A = X_p X_p^T  (M = 128, N = 128, K = 256)
      if (threadIdx.x == 0 && cx.ok) mma_x3(tA, x_hi, x_lo, rgsN, x_hi, x_lo, rgsN, 0, R2, R2, NH);
      pair_commit_wait(cx);
      float af[64];   // this thread's row, columns [64 half, 64 half + 64) of A
      tc::tmem_ld16(tA + lane_base + 64 * half, af);
      tc::tmem_ld16(tA + lane_base + 64 * half + 16, af + 16);
      tc::tmem_ld16(tA + lane_base + 64 * half + 32, af + 32);
      tc::tmem_ld16(tA + lane_base + 64 * half + 48, af + 48);
      tc::tmem_ld_wait();
      // stage this CTA's packed partial (row < 64 with half 1 holds block
      // (0, 1); half 0 the lower triangle of block (0, 0); rows >= 64 with
      // half 1 the upper triangle of block (1, 1); block (1, 0) is not sent)
      {
        float* q = stg + 64 * 64;
        const int r1 = row & 63;
        if (row < 64 && half == 1) {
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4)
            *reinterpret_cast<float4*>(stg + xswz64(row, 4 * q4)) =
                make_float4(af[4 * q4], af[4 * q4 + 1], af[4 * q4 + 2], af[4 * q4 + 3]);
        } else if (row < 64) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (j <= r1) q[r1 * kQS + j] = af[j];
        } else if (half == 1) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (j >= r1) q[r1 * kQS + j + 1] = af[j];
        }
      }
      tc::fence_smem_to_async();   // staging is the bulk copy's source
      __syncthreads();
      // one copy once the partner's A/B' buffer is free (it arrives on
      // xfree when its B'X product is done)
      bool good = true;
      if (threadIdx.x == 0 && cx.ok) {
        good = tc::mbar_wait(&xfree, xe & 1, kWaitCycles);
        if (good) {
          const uint32_t xb = mapa2(tc::smem_u32(&xdata), p ^ 1u);
          bulk_to_partner(mapa2(tc::smem_u32(recv), p ^ 1u), tc::smem_u32(stg), kPartBytes, xb);
          good = tc::mbar_wait(&xdata, xe & 1, kWaitCycles);
          if (good) mbar_arm_tx2(&xdata, kPartBytes);   // the next exchange
          bulk_wait_read2();   // staging read: it may be rewritten
        }
      }
      ++xe;
      if (__syncthreads_or(!good)) cx.ok = false;
      {
        // partner's entries of my row, columns [64 half, 64 half + 64)
        const float* rq = recv + 64 * 64;
        const int r1 = row & 63;
        if (row < 64 && half == 1) {
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 o = *reinterpret_cast<const float4*>(recv + xswz64(row, 4 * q4));
            af[4 * q4] += o.x; af[4 * q4 + 1] += o.y; af[4 * q4 + 2] += o.z; af[4 * q4 + 3] += o.w;
          }
        } else if (row < 64) {
          // block (0, 0): the stored triangle up to the diagonal, the rest
          // from the rows below it (P00[r][j] = P00[j][r])
#pragma unroll
          for (int j = 0; j < 64; ++j) af[j] += rq[j <= r1 ? r1 * kQS + j : j * kQS + r1];
        } else if (half == 0) {
          // block (1, 0): the transpose of block (0, 1)
#pragma unroll
          for (int j = 0; j < 64; ++j) af[j] += recv[xswz64(j, r1)];
        } else {
          // block (1, 1): the stored triangle from the diagonal on, the rest
          // from the rows above it (P11[r][j] = P11[j][r])
#pragma unroll
          for (int j = 0; j < 64; ++j) af[j] += rq[j >= r1 ? r1 * kQS + j + 1 : j * kQS + r1 + 1];
        }
      }
      if (it == 0) {
        // this thread's diagonal entry of A (if its columns hold one), summed
        // over the CTA: trace(A) = ||Shat||^2 (both CTAs hold the same
        // diagonal, so both get the same s)
        const int jd = row - 64 * half;
        float dg = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) dg = (j == jd) ? af[j] : dg;
        for (int o = 16; o > 0; o >>= 1) dg += __shfl_xor_sync(0xffffffffu, dg, o);
        if (lane == 0) red[warp] = dg;
      }
      __syncthreads();   // every received entry read before the buffer takes A hi/lo
      if (it == 0) {
        float tot = 0.f;
        for (int k2 = 0; k2 < NT2 / 32; ++k2) tot += red[k2];
        scale = lam / (lam * sqrtf(tot) + kNsEps);
        const float s2 = scale * scale;
#pragma unroll
        for (int j = 0; j < 64; ++j) af[j] *= s2;
      }
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) store_split16(a_hi, a_lo, tc::core_offset(row, 64 * half + 8 * q8, rgsR), af + 8 * q8);
      sync_for_mma();
      // A^2 (symmetric A: rows serve as the K-major B operand)
      if (threadIdx.x == 0 && cx.ok) mma_x3(tA2, a_hi, a_lo, rgsR, a_hi, a_lo, rgsR, 0, R2, R2, R2);
      pair_commit_wait(cx);
      for (int q = 0; q < 64; q += 16) {
        float a2[16];
        tc::tmem_ld16(tA2 + lane_base + 64 * half + q, a2);
        tc::tmem_ld_wait();
        float bp[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          bp[j] = kNsB * af[q + j] + kNsC * a2[j] + (row == 64 * half + q + j ? kNsA : 0.f);
        store_split16(a_hi, a_lo, tc::core_offset(row, 64 * half + q, rgsR), bp);
        store_split16(a_hi, a_lo, tc::core_offset(row, 64 * half + q + 8, rgsR), bp + 8);
      }
      sync_for_mma();
      // X_p <- B' X_p  (M = 128, N = 256, K = 128; X read as MN-major)
      if (threadIdx.x == 0 && cx.ok) mma_x3(tX, a_hi, a_lo, rgsR, x_hi, x_lo, rgsN, 1, R2, NH, R2);
      pair_commit_wait(cx);
      const bool last = (it == g.ns_iters - 1);
      // B' is consumed: the partner may send the next exchange
      if (!last && threadIdx.x == 0 && cx.ok) mbar_arrive_remote(xfree_peer);
      // U rows go out through shared memory, one bulk copy per row (a
      // thread's own row stored straight to global memory would touch 32
      // lines per warp store); the staging spans the X and A/B' buffers,
      // which nothing touches until this CTA's next momentum product
      float* ust = reinterpret_cast<float*>(sm);
      for (int c32 = 32 * half; c32 < NH; c32 += 64) {
        float v[32];
        tc::tmem_ld16(tX + lane_base + c32, v);
        tc::tmem_ld16(tX + lane_base + c32 + 16, v + 16);
        tc::tmem_ld_wait();
        if (it == 0) {
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] *= scale;   // X_1 = s B' Shat
        }
        if (last) {
          float4* o = reinterpret_cast<float4*>(ust + row * kUS + c32);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) store_split16(x_hi, x_lo, tc::core_offset(row, c32 + 8 * q8, rgsN), v + 8 * q8);
        }
      }
      if (last) {
        tc::fence_smem_to_async();
        __syncthreads();
        if (threadIdx.x < R2 && cx.ok) {
          bulk_to_global(slot + (size_t)threadIdx.x * n + p * NH, tc::smem_u32(ust + threadIdx.x * kUS), NH * 4);
          bulk_wait_read2();   // the staging is rewritten by the next token
        }
      }
      sync_for_mma();
    }
  }
  if (threadIdx.x < R2) bulk_wait_all2();   // the exchange copies and the U rows
  if (!cx.ok && threadIdx.x == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync2();
  if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

// transpose every unit's rows x cols matrix into cols x rows
__global__ void k_transpose_units(const float* __restrict__ in, float* __restrict__ out, int rows, int cols) {
  __shared__ float tile[32][33];
  const int u = blockIdx.z;
  const float* src = in + (size_t)u * rows * cols;
  float* dst = out + (size_t)u * rows * cols;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = src[(size_t)r * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) dst[(size_t)c * rows + r] = tile[threadIdx.x][i];
  }
}

// 0: not covered; 1: short side 64 (one CTA per task); 2: 128 x 512 (CTA pairs)
int ns_tc_kind(const Geom& g) {
  if (g.ns_iters <= 0 || g.ns_target != ATLAS_NS_MOMENTUM) return 0;
  const int Kp = (g.Kw + 15) / 16 * 16;
  if (Kp > 128) return 0;
  int kind = -1, n0 = -1;
  for (int m = 0; m < g.nmat; ++m) {
    const int s = g.rows[m] < g.cols[m] ? g.rows[m] : g.cols[m];
    const int l = g.rows[m] < g.cols[m] ? g.cols[m] : g.rows[m];
    int k = 0;
    if (s == R && l % 16 == 0 && l <= 256) k = 1;
    if (s == R2 && l == 2 * NH && Kp <= 96) k = 2;
    if (!k || (kind >= 0 && k != kind) || (n0 >= 0 && l != n0)) return 0;
    kind = k;
    n0 = l;
  }
  if (kind == 1 && ns_smem_layout(n0, Kp).total > 226 * 1024) return 0;
  return kind;
}

bool ns_tc_supported(const Geom& g) { return ns_tc_kind(g) != 0; }

// momentum state of the tensor-core path: transposed (X orientation) for
// matrices with rows > cols
cudaError_t ns_tc_state_in(const Geom& g, int m, const float* src, float* dst, cudaStream_t st) {
  const size_t bytes = (size_t)g.units * g.rows[m] * g.cols[m] * sizeof(float);
  if (g.rows[m] <= g.cols[m]) return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  dim3 grid((g.cols[m] + 31) / 32, (g.rows[m] + 31) / 32, g.units);
  k_transpose_units<<<grid, dim3(32, 8), 0, st>>>(src, dst, g.rows[m], g.cols[m]);
  return cudaGetLastError();
}

cudaError_t ns_tc_state_out(const Geom& g, int m, const float* src, float* dst, cudaStream_t st) {
  const size_t bytes = (size_t)g.units * g.rows[m] * g.cols[m] * sizeof(float);
  if (g.rows[m] <= g.cols[m]) return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  dim3 grid((g.rows[m] + 31) / 32, (g.cols[m] + 31) / 32, g.units);
  k_transpose_units<<<grid, dim3(32, 8), 0, st>>>(src, dst, g.cols[m], g.rows[m]);
  return cudaGetLastError();
}

cudaError_t ns_tc_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, size_t slot_stride, int num_sms,
                         const float* theta, const float* eta, cudaStream_t st) {
  const int n = g.rows[0] < g.cols[0] ? g.cols[0] : g.rows[0];
  const int Kp = (g.Kw + 15) / 16 * 16;
  if (ns_tc_kind(g) == 2) {
    cudaError_t e = cudaFuncSetAttribute(k_ns_tc128, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM2);
    if (e != cudaSuccess) return e;
    const int ntasks = g.units * g.nmat * (ch.e - ch.s - ns_first_row(g, ch));
    int ncl = num_sms / 2;
    if (ncl > ntasks) ncl = ntasks;
    k_ns_tc128<<<2 * ncl, NT2, SMEM2, st>>>(g, ch, w, buf, slot_stride, Kp, theta, eta);
    return cudaGetLastError();
  }
  const int smem = ns_smem_layout(n, Kp).total;
  cudaFuncSetAttribute(k_ns_tc64, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int ntasks = g.units * g.nmat * (ch.e - ch.s - ns_first_row(g, ch));
  const int grid = ntasks < num_sms ? ntasks : num_sms;   // each CTA takes a contiguous run of tasks
  k_ns_tc64<<<grid, NT, smem, st>>>(g, ch, w, buf, slot_stride, n, Kp);
  return cudaGetLastError();
}

}  // namespace atlas
