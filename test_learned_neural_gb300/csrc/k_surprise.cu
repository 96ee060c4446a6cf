// Newton-Schulz on the windowed surprise (atlas-torch README, "Atlas
// Extensions": Muon / Newton-Schulz orthogonalises the surprise updates; the
// per-token store path keeps eta outside Newton-Schulz):
//
//   S_t = eta_t S_{t-1} - theta_t NS(g_t),   W_t = (1 - alpha_t) W_{t-1} + S_t,
//
// with g_t the gamma-weighted sum of the per-token gradients of the last c
// tokens at the chunk-start weights.  Per matrix, g_t = L_t^T R_t: the rows
// of L are the window's memory inputs (x_i, or a_i for W2), the rows of R
// the output-side factors (dz_i or dy_i, 2 gamma_i folded in).  Every
// Newton-Schulz iterate keeps that form, X = L^T K R with a c x c core K:
//
//   X X^T X = L^T K H R,   H = Gr K^T Gl K,   Gl = L L^T,  Gr = R R^T,
//   X <- a X + b X X^T X + c (X X^T)^2 X   becomes   K <- K (a I + b H + c H^2),
//
// starting from K = I / (|g|_F + eps) with |g|_F^2 = sum(Gl (.) Gr).  This is
// the same iteration exactly (not an approximation), on c x c matrices.
//
// The momentum and weights then stay in dual form over the chunk's window
// rows, with banded (bandwidth c) coefficient matrices instead of the
// diagonal ones of the plain rule:
//
//   S_t = A_t Sbar - L^T Ms_t R,      Ms_t = eta_t Ms_{t-1} + theta_t K~_t,
//   W_t = B_t Wbar + D_t Sbar - L^T Mw_t R,   Mw_t = (1 - alpha_t) Mw_{t-1} + Ms_t,
//
// K~_t being K_t placed on token t's window rows.  The read-out of token t
// goes through (r_t L^T) Mw_t R; the chunk-end state through L^T (Ms_e R).
#include "atlas_common.cuh"
#include "simt_tile.cuh"

namespace atlas {
namespace {

constexpr float kNsA = 3.4445f, kNsB = -4.7750f, kNsC = 2.0315f, kNsEps = 1e-7f;

// floats per unit of the scratch, by part
struct SurpLayout {
  size_t gram;   // [nmat][2][Kw][2c-1]  band of L L^T, R R^T
  size_t kt;     // [nmat][C][c][c]      c x c cores
  size_t mwb;    // [nmat][C][Kw][2c-1]  band of the read-out's Mw (token t's, or t-1's before the update)
  size_t mse;    // [nmat][Kw][2c-1]     band of Ms at the chunk end
  size_t mwe;    // [nmat][Kw][2c-1]     band of Mw at the chunk end
  size_t rp;     // [nmat][2][Kw][maxcols]  Ms_e R, Mw_e R
  size_t g2;     // [2][64][kwp] bf16 hi, then lo: the read-outs' (G Mw) tiles (tensor-core path)
  size_t per_unit;
};

__host__ __device__ inline int max_cols(const Geom& g) {
  return g.nmat > 1 && g.cols[1] > g.cols[0] ? g.cols[1] : g.cols[0];
}

__host__ __device__ inline SurpLayout surp_layout(const Geom& g) {
  const size_t Kw = g.Kw, c = g.c, band = 2 * c - 1, nm = g.nmat;
  SurpLayout L;
  size_t o = 0;
  L.gram = o; o += nm * 2 * Kw * band;
  L.kt = o;   o += nm * g.C * c * c;
  L.mwb = o;  o += nm * g.C * Kw * band;
  L.mse = o;  o += nm * Kw * band;
  L.mwe = o;  o += nm * Kw * band;
  L.rp = o;   o += nm * 2 * Kw * (size_t)max_cols(g);
  L.g2 = o;   o += 2 * 64 * ((Kw + 15) / 16 * 16);
  L.per_unit = o;
  return L;
}

// window rows i (token lo + i) of matrix m's factors; widths rows[m], cols[m]
__device__ __forceinline__ const float* lfac(const Geom& g, const Chunk& ch, const Work& w, int u, int m) {
  if (g.depth == 2 && m == 1) return w.Aact + (size_t)u * g.Kw * g.hidden;
  return w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
}
__device__ __forceinline__ const float* rfac(const Geom& g, const Work& w, int u, int m) {
  if (g.depth == 2 && m == 0) return w.DZ + (size_t)u * g.Kw * g.hidden;
  return w.DY + (size_t)u * g.Kw * g.d_v;
}

// token t's window: rows [lo_w, hi_w] of the chunk's window rows
__device__ __forceinline__ void window_rows(const Geom& g, const Chunk& ch, int t, int& lo_w, int& hi_w) {
  lo_w = (t - g.c + 1 > ch.lo ? t - g.c + 1 : ch.lo) - ch.lo;
  hi_w = t - ch.lo;
}

// band of L L^T (side 0) and R R^T (side 1); one block per (row i, matrix
// and side, unit), one warp per band offset
__global__ void __launch_bounds__(256) k_surp_gram(Geom g, Chunk ch, Work w) {
  const int i = blockIdx.x, m = blockIdx.y >> 1, side = blockIdx.y & 1, u = blockIdx.z;
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1;
  const float* P = side ? rfac(g, w, u, m) : lfac(g, ch, w, u, m);
  const int width = side ? g.cols[m] : g.rows[m];
  float* out = w.surp + (size_t)u * S.per_unit + S.gram + (((size_t)m * 2 + side) * g.Kw + i) * band;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int d = warp; d < band; d += blockDim.x / 32) {
    const int j = i + d - (g.c - 1);
    float acc = 0.f;
    if (j >= 0 && j < ch.nw)
      for (int k = lane; k < width; k += 32) acc += P[(size_t)i * width + k] * P[(size_t)j * width + k];
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) out[d] = acc;
  }
}

// c x c Newton-Schulz core of token r of the chunk, matrix m, unit u: one
// warp per (token, matrix), eight per block; the warp's six n x n work
// matrices (n <= c <= 32, row stride c + 1) sit in its own slice of
// shared memory and its steps synchronise with __syncwarp only.
__global__ void __launch_bounds__(256) k_surp_ns(Geom g, Chunk ch, Work w) {
  extern __shared__ float ns_sm[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r = blockIdx.x * 8 + warp, m = blockIdx.y, u = blockIdx.z, t = ch.s + r;
  if (r >= ch.e - ch.s) return;   // whole warps leave; no block-wide barrier follows
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1, c = g.c, ld = c + 1, sz = c * ld;
  float* Gl = ns_sm + (size_t)warp * 6 * sz;
  float* Gr = Gl + sz;
  float* K = Gr + sz;
  float* T1 = K + sz;
  float* T2 = T1 + sz;
  float* H = T2 + sz;
  int lo_w, hi_w;
  window_rows(g, ch, t, lo_w, hi_w);
  const int n = hi_w - lo_w + 1;   // rows of this token's window (<= c)
  const float* gb = w.surp + (size_t)u * S.per_unit + S.gram + (size_t)m * 2 * g.Kw * band;
  float part = 0.f;
  for (int e = lane; e < n * n; e += 32) {
    const int a = e / n, b = e % n;
    const int d = b - a + c - 1;
    const float gl = gb[(size_t)(lo_w + a) * band + d];
    const float gr = gb[((size_t)g.Kw + lo_w + a) * band + d];
    Gl[a * ld + b] = gl;
    Gr[a * ld + b] = gr;
    part += gl * gr;
  }
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  const float nrm = sqrtf(fmaxf(part, 0.f));
  // |g|_F = 0: the surprise is zero and so is its orthogonalisation
  const float k0 = nrm > 0.f ? 1.f / (nrm + kNsEps) : 0.f;
  for (int e = lane; e < n * n; e += 32) {
    const int a = e / n, b = e % n;
    K[a * ld + b] = a == b ? k0 : 0.f;
  }
  __syncwarp();
  for (int it = 0; it < g.ns_iters; ++it) {
    // T1 = Gl K, T2 = K^T T1, H = Gr T2, T1 = H H, T2 = a I + b H + c H^2, K = K T2
    for (int e = lane; e < n * n; e += 32) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += Gl[a * ld + k] * K[k * ld + b];
      T1[a * ld + b] = acc;
    }
    __syncwarp();
    for (int e = lane; e < n * n; e += 32) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += K[k * ld + a] * T1[k * ld + b];
      T2[a * ld + b] = acc;
    }
    __syncwarp();
    for (int e = lane; e < n * n; e += 32) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += Gr[a * ld + k] * T2[k * ld + b];
      H[a * ld + b] = acc;
    }
    __syncwarp();
    for (int e = lane; e < n * n; e += 32) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += H[a * ld + k] * H[k * ld + b];
      T2[a * ld + b] = (a == b ? kNsA : 0.f) + kNsB * H[a * ld + b] + kNsC * acc;
    }
    __syncwarp();
    for (int e = lane; e < n * n; e += 32) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += K[a * ld + k] * T2[k * ld + b];
      T1[a * ld + b] = acc;
    }
    __syncwarp();
    for (int e = lane; e < n * n; e += 32) {
      const int a = e / n, b = e % n;
      K[a * ld + b] = T1[a * ld + b];
    }
    __syncwarp();
  }
  float* kt = w.surp + (size_t)u * S.per_unit + S.kt + ((size_t)m * g.C + r) * c * c;
  for (int e = lane; e < c * c; e += 32) {
    const int a = e / c, b = e % c;
    kt[e] = (a < n && b < n) ? K[a * ld + b] : 0.f;
  }
}

// banded coefficient scans over the chunk; one thread per band element
__global__ void __launch_bounds__(256) k_surp_scan(Geom g, Chunk ch, Work w, const float* theta, const float* eta,
                                                   const float* alpha) {
  const int m = blockIdx.y, u = blockIdx.z;
  const int band = 2 * g.c - 1, c = g.c;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= g.Kw * band) return;
  const int i = e / band, d = e % band, j = i + d - (c - 1);
  const bool valid = i < ch.nw && j >= 0 && j < ch.nw;
  const SurpLayout S = surp_layout(g);
  float* base = w.surp + (size_t)u * S.per_unit;
  const float* kt = base + S.kt + (size_t)m * g.C * c * c;
  float* mwb = base + S.mwb + (size_t)m * g.C * g.Kw * band;
  const bool pre = g.readout == ATLAS_READOUT_PRE;
  float Ms = 0.f, Mw = 0.f;
  for (int r = 0; r < ch.e - ch.s; ++r) {
    const int t = ch.s + r;
    int lo_w, hi_w;
    window_rows(g, ch, t, lo_w, hi_w);
    const bool in = valid && i >= lo_w && i <= hi_w && j >= lo_w && j <= hi_w;
    const float kv = in ? kt[(size_t)r * c * c + (i - lo_w) * c + (j - lo_w)] : 0.f;
    const size_t gi = (size_t)u * g.T + t;
    Ms = eta[gi] * Ms + theta[gi] * kv;
    const float Mw_prev = Mw;
    Mw = (1.f - alpha[gi]) * Mw + Ms;
    mwb[((size_t)r * g.Kw + i) * band + d] = pre ? Mw_prev : Mw;   // the weights token t reads out
  }
  base[S.mse + ((size_t)m * g.Kw + i) * band + d] = Ms;
  base[S.mwe + ((size_t)m * g.Kw + i) * band + d] = Mw;
}

constexpr int TG = 8;   // tokens per read-out block: W, S columns are loaded once for all of them

// read-out of tokens [r0, r0 + TG): y = B_t r W + D_t r S - ((r L^T) Mw_t) R
// (through the MLP at depth 2); one block per (token group, unit)
__global__ void __launch_bounds__(256) k_surp_readout(Geom g, Chunk ch, Work w, int buf, float* y) {
  extern __shared__ float sm[];
  __shared__ float Bt[TG], Dt[TG];
  const int u = blockIdx.y, r0 = blockIdx.x * TG;
  const int Ct = ch.e - ch.s, nt = Ct - r0 < TG ? Ct - r0 : TG, nw = ch.nw;
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1, F = g.F, Kw = g.Kw;
  float* rs = sm;              // [TG][F]
  float* gm = rs + TG * F;     // [TG][Kw]
  float* gm2 = gm + TG * Kw;   // [TG][Kw]
  float* aq = gm2 + TG * Kw;   // [TG][hidden] (depth 2)
  for (int e = threadIdx.x; e < TG * F; e += blockDim.x) {
    const int tt = e / F, f = e % F;
    rs[e] = tt < nt ? w.R[((size_t)u * g.T + ch.s + r0 + tt) * F + f] : 0.f;
  }
  if (threadIdx.x < TG) {
    const int rr = (g.readout == ATLAS_READOUT_PRE ? -1 : 0) + r0 + (int)threadIdx.x;
    const bool ok = rr >= 0 && r0 + (int)threadIdx.x < Ct;
    Bt[threadIdx.x] = ok ? w.Bp[(size_t)u * g.C + rr] : (rr < 0 ? 1.f : 0.f);
    Dt[threadIdx.x] = ok ? w.Dp[(size_t)u * g.C + rr] : 0.f;
  }
  __syncthreads();
  const float* mwb = w.surp + (size_t)u * S.per_unit + S.mwb;
  // gm[tt][i] = r . L_i, then gm2[tt][j] = sum_i gm[tt][i] Mw_t[i][j] (band)
  auto mix = [&](const float* Lw, int width, const float* vec, int vstride, const float* Mw) {
    // one warp per window row: coalesced loads of L_i, all TG tokens at once
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int i = warp; i < nw; i += blockDim.x / 32) {
      float acc[TG];
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) acc[tt] = 0.f;
#pragma unroll 4
      for (int f = lane; f < width; f += 32) {
        const float lv = Lw[(size_t)i * width + f];
#pragma unroll
        for (int tt = 0; tt < TG; ++tt) acc[tt] += vec[tt * vstride + f] * lv;
      }
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) {
        float v = acc[tt];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) gm[tt * Kw + i] = v;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < TG * nw; e += blockDim.x) {
      const int tt = e / nw, j = e % nw;
      float acc = 0.f;
      if (tt < nt) {
        const float* M = Mw + (size_t)(r0 + tt) * Kw * band;
        const int i0 = j - g.c + 1 > 0 ? j - g.c + 1 : 0, i1 = j + g.c - 1 < nw - 1 ? j + g.c - 1 : nw - 1;
        for (int i = i0; i <= i1; ++i) acc += gm[tt * Kw + i] * M[(size_t)i * band + (j - i + g.c - 1)];
      }
      gm2[tt * Kw + j] = acc;
    }
    __syncthreads();
  };
  // out[tt][k] = B_t (v W)[k] + D_t (v S)[k] - (gm2 R)[k] for k < cols
  auto terms = [&](const float* vec, int vstride, int K, const float* Wm, const float* Sm, const float* Rf, int cols,
                   int k, float* res) {
    float a[TG], b[TG], c2[TG];
#pragma unroll
    for (int tt = 0; tt < TG; ++tt) a[tt] = b[tt] = c2[tt] = 0.f;
    // unrolled 16 deep so that many W, S loads are in flight per thread (the
    // loop is bound by their latency, not by the FMAs)
#pragma unroll 16
    for (int f = 0; f < K; ++f) {
      const float wv = Wm[(size_t)f * cols + k], sv = Sm[(size_t)f * cols + k];
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) {
        a[tt] += vec[tt * vstride + f] * wv;
        b[tt] += vec[tt * vstride + f] * sv;
      }
    }
#pragma unroll 16
    for (int j = 0; j < nw; ++j) {
      const float rv = Rf[(size_t)j * cols + k];
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) c2[tt] += gm2[tt * Kw + j] * rv;
    }
#pragma unroll
    for (int tt = 0; tt < TG; ++tt) res[tt] = Bt[tt] * a[tt] + Dt[tt] * b[tt] - c2[tt];
  };
  mix(lfac(g, ch, w, u, 0), F, rs, F, mwb);
  if (g.depth == 1) {
    const float* W = w.Wst[buf][0] + (size_t)u * F * g.d_v;
    const float* Sb = w.Sst[buf][0] + (size_t)u * F * g.d_v;
    for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
      float res[TG];
      terms(rs, F, F, W, Sb, rfac(g, w, u, 0), g.d_v, k, res);
      for (int tt = 0; tt < nt; ++tt) y[((size_t)u * g.T + ch.s + r0 + tt) * g.d_v + k] = res[tt];
    }
    return;
  }
  const int h = g.hidden;
  for (int k = threadIdx.x; k < h; k += blockDim.x) {
    float res[TG];
    terms(rs, F, F, w.Wst[buf][0] + (size_t)u * F * h, w.Sst[buf][0] + (size_t)u * F * h, rfac(g, w, u, 0), h, k,
          res);
#pragma unroll
    for (int tt = 0; tt < TG; ++tt) aq[tt * h + k] = siluf_(res[tt]);
  }
  __syncthreads();
  mix(lfac(g, ch, w, u, 1), h, aq, h, mwb + (size_t)g.C * Kw * band);
  for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
    float res[TG];
    terms(aq, h, h, w.Wst[buf][1] + (size_t)u * h * g.d_v, w.Sst[buf][1] + (size_t)u * h * g.d_v,
          rfac(g, w, u, 1), g.d_v, k, res);
    for (int tt = 0; tt < nt; ++tt)
      y[((size_t)u * g.T + ch.s + r0 + tt) * g.d_v + k] = rs[tt * F + k] + res[tt];
  }
}

// Ms_e R and Mw_e R (rows i of the window) of matrix m
__global__ void __launch_bounds__(256) k_surp_rprime(Geom g, Chunk ch, Work w) {
  // One block per (128-column block, matrix, unit): the block's columns of R
  // (window rows 0 .. nw - 1) and both band matrices are staged in shared
  // memory once, so each R row is read from global memory once instead of
  // once per band row that uses it; thread (which, column) then forms its
  // column for every window row i, in the same order of terms.
  extern __shared__ float rp_sm[];   // R block [nw][128], then bands [2][nw][2c - 1]
  const int cb0 = blockIdx.x * 128, m = blockIdx.y, u = blockIdx.z;
  const int cols = g.cols[m];
  if (cb0 >= cols) return;
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1, c = g.c, nw = ch.nw, mc = max_cols(g);
  const int ncol = cols - cb0 < 128 ? cols - cb0 : 128;
  const float* R = rfac(g, w, u, m);
  const float* base = w.surp + (size_t)u * S.per_unit;
  float* Rs = rp_sm;
  float* Ms = rp_sm + nw * 128;
  // asynchronous 4-byte copies, all in flight at once (columns past the
  // matrix are zero-filled: source size 0)
  for (int e = threadIdx.x; e < nw * 128; e += blockDim.x) {
    const int j = e / 128, b = e % 128;
    const float* src = R + (size_t)j * cols + cb0 + (b < ncol ? b : 0);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(Rs + e)),
                 "l"(src), "r"(b < ncol ? 4 : 0)
                 : "memory");
  }
  for (int e = threadIdx.x; e < 2 * nw * band; e += blockDim.x) {
    const int wh = e / (nw * band), r = e % (nw * band);
    const float* src = base + (wh ? S.mwe : S.mse) + (size_t)m * g.Kw * band + r;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(Ms + e)), "l"(src)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  const int which = threadIdx.x / 128, b = threadIdx.x % 128;
  if (which > 1 || b >= ncol) return;
  const float* M = Ms + which * nw * band;
  float* out = w.surp + (size_t)u * S.per_unit + S.rp + ((size_t)m * 2 + which) * g.Kw * mc + cb0 + b;
  for (int i = 0; i < nw; ++i) {
    const int j0 = i - c + 1 > 0 ? i - c + 1 : 0, j1 = i + c - 1 < nw - 1 ? i + c - 1 : nw - 1;
    float acc = 0.f;
    for (int j = j0; j <= j1; ++j) acc += M[i * band + (j - i + c - 1)] * Rs[j * 128 + b];
    out[(size_t)i * mc] = acc;
  }
}

// chunk-end state: S = A_e Sbar - L^T (Ms_e R), W = B_e Wbar + D_e Sbar - L^T (Mw_e R);
// one 64 x 64 tile of matrix m per block
__global__ void __launch_bounds__(256) k_surp_state(Geom g, Chunk ch, Work w, int m, int buf) {
  __shared__ float As[16 * 64], Bs[16 * 64];
  const int u = blockIdx.z, a0 = blockIdx.y * 64, b0 = blockIdx.x * 64;
  const int rows = g.rows[m], cols = g.cols[m], mc = max_cols(g);
  const SurpLayout S = surp_layout(g);
  const float* L = lfac(g, ch, w, u, m);
  const float* rps = w.surp + (size_t)u * S.per_unit + S.rp + ((size_t)m * 2 + 0) * g.Kw * mc;
  const float* rpw = rps + (size_t)g.Kw * mc;
  float accs[4][4], accw[4][4];
  tile_gemm(TileOp{L, 1, rows}, TileOp{rps, 1, mc}, rows, cols, ch.nw, a0, b0, accs, As, Bs);
  tile_gemm(TileOp{L, 1, rows}, TileOp{rpw, 1, mc}, rows, cols, ch.nw, a0, b0, accw, As, Bs);
  const int re = ch.e - 1 - ch.s;
  const float Ae = w.Ap[(size_t)u * g.C + re], Be = w.Bp[(size_t)u * g.C + re], De = w.Dp[(size_t)u * g.C + re];
  const size_t n = (size_t)rows * cols;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int p = 0; p < 4; ++p) {
    const int a = a0 + ty * 4 + p;
    if (a >= rows) continue;
    for (int q = 0; q < 4; ++q) {
      const int b = b0 + tx * 4 + q;
      if (b >= cols) continue;
      const size_t o = (size_t)u * n + (size_t)a * cols + b;
      const float Sb = w.Sst[buf][m][o], Wb = w.Wst[buf][m][o];
      w.Sst[buf ^ 1][m][o] = Ae * Sb - accs[p][q];
      w.Wst[buf ^ 1][m][o] = Be * Wb + De * Sb - accw[p][q];
    }
  }
}

}  // namespace

static cudaError_t rprime_launch(const Geom& g, const Chunk& ch, const Work& w, cudaStream_t st) {
  const int sm = (ch.nw * 128 + 2 * ch.nw * (2 * g.c - 1)) * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_surp_rprime, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
  if (e != cudaSuccess) return e;
  k_surp_rprime<<<dim3((max_cols(g) + 127) / 128, g.nmat, g.units), 256, sm, st>>>(g, ch, w);
  return cudaGetLastError();
}

size_t surprise_floats(const Geom& g, size_t units) { return units * surp_layout(g).per_unit; }

SurpOff surprise_offsets(const Geom& g) {
  const SurpLayout L = surp_layout(g);
  SurpOff so;
  so.per_unit = L.per_unit;
  so.mwb = L.mwb;
  so.rp = L.rp;
  so.g2 = L.g2;
  so.maxcols = max_cols(g);
  return so;
}

cudaError_t surprise_chunk(const Geom& g, const Chunk& ch, const Work& w, const float* theta, const float* eta,
                           const float* alpha, float* y, int buf, cudaStream_t st, int* nl) {
  const int Ct = ch.e - ch.s, band = 2 * g.c - 1;
  k_surp_gram<<<dim3(ch.nw, g.nmat * 2, g.units), 256, 0, st>>>(g, ch, w);
  const int nsm = 8 * 6 * g.c * (g.c + 1) * (int)sizeof(float);   // eight warps' work matrices
  cudaError_t es = cudaFuncSetAttribute(k_surp_ns, cudaFuncAttributeMaxDynamicSharedMemorySize, nsm);
  if (es != cudaSuccess) return es;
  k_surp_ns<<<dim3((Ct + 7) / 8, g.nmat, g.units), 256, nsm, st>>>(g, ch, w);
  k_surp_scan<<<dim3((g.Kw * band + 255) / 256, g.nmat, g.units), 256, 0, st>>>(g, ch, w, theta, eta, alpha);
  if (surprise_tc_supported(g)) {
    // tensor cores: read-out in two launches (hidden read-out, output), the
    // chunk-end state of both matrices in one
    cudaError_t e = surprise_tc_readout(g, ch, w, buf, y, st);
    if (e != cudaSuccess) return e;
    e = rprime_launch(g, ch, w, st);
    if (e != cudaSuccess) return e;
    e = surprise_tc_state(g, ch, w, buf, st);
    if (e != cudaSuccess) return e;
    *nl += 9;
    return cudaGetLastError();
  }
  const size_t sr = (size_t)TG * (g.F + 2 * g.Kw + (g.depth == 2 ? g.hidden : 0)) * sizeof(float);
  cudaFuncSetAttribute(k_surp_readout, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sr);
  k_surp_readout<<<dim3((Ct + TG - 1) / TG, g.units), 256, sr, st>>>(g, ch, w, buf, y);
  cudaError_t e = rprime_launch(g, ch, w, st);
  if (e != cudaSuccess) return e;
  for (int m = 0; m < g.nmat; ++m)
    k_surp_state<<<dim3((g.cols[m] + 63) / 64, (g.rows[m] + 63) / 64, g.units), 256, 0, st>>>(g, ch, w, m, buf);
  *nl += 5 + g.nmat;
  return cudaGetLastError();
}

}  // namespace atlas
