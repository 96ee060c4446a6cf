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

// c x c Newton-Schulz core of token r of the chunk, matrix m, unit u
__global__ void __launch_bounds__(256) k_surp_ns(Geom g, Chunk ch, Work w) {
  __shared__ float Gl[32][33], Gr[32][33], K[32][33], T1[32][33], T2[32][33], H[32][33];
  __shared__ float red[8];
  const int r = blockIdx.x, m = blockIdx.y, u = blockIdx.z, t = ch.s + r;
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1, c = g.c;
  int lo_w, hi_w;
  window_rows(g, ch, t, lo_w, hi_w);
  const int n = hi_w - lo_w + 1;   // rows of this token's window (<= c)
  const float* gb = w.surp + (size_t)u * S.per_unit + S.gram + (size_t)m * 2 * g.Kw * band;
  float part = 0.f;
  for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
    const int a = e / n, b = e % n;
    const int d = b - a + c - 1;
    const float gl = gb[(size_t)(lo_w + a) * band + d];
    const float gr = gb[((size_t)g.Kw + lo_w + a) * band + d];
    Gl[a][b] = gl;
    Gr[a][b] = gr;
    part += gl * gr;
  }
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = part;
  __syncthreads();
  float s2 = 0.f;
  for (int k = 0; k < (int)(blockDim.x / 32); ++k) s2 += red[k];
  const float nrm = sqrtf(fmaxf(s2, 0.f));
  // |g|_F = 0: the surprise is zero and so is its orthogonalisation
  const float k0 = nrm > 0.f ? 1.f / (nrm + kNsEps) : 0.f;
  for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
    const int a = e / n, b = e % n;
    K[a][b] = a == b ? k0 : 0.f;
  }
  __syncthreads();
  for (int it = 0; it < g.ns_iters; ++it) {
    // T1 = Gl K, T2 = K^T T1, H = Gr T2, T1 = H H, T2 = a I + b H + c H^2, K = K T2
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += Gl[a][k] * K[k][b];
      T1[a][b] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += K[k][a] * T1[k][b];
      T2[a][b] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += Gr[a][k] * T2[k][b];
      H[a][b] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += H[a][k] * H[k][b];
      T2[a][b] = (a == b ? kNsA : 0.f) + kNsB * H[a][b] + kNsC * acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
      const int a = e / n, b = e % n;
      float acc = 0.f;
      for (int k = 0; k < n; ++k) acc += K[a][k] * T2[k][b];
      T1[a][b] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
      const int a = e / n, b = e % n;
      K[a][b] = T1[a][b];
    }
    __syncthreads();
  }
  float* kt = w.surp + (size_t)u * S.per_unit + S.kt + ((size_t)m * g.C + r) * c * c;
  for (int e = threadIdx.x; e < c * c; e += blockDim.x) {
    const int a = e / c, b = e % c;
    kt[e] = (a < n && b < n) ? K[a][b] : 0.f;
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

// out_j = sum_i v_i M[i][j] over the band (M rows of 2c - 1 entries)
__device__ void band_mix(const Geom& g, int nw, const float* v, const float* M, float* out) {
  const int band = 2 * g.c - 1, c = g.c;
  for (int j = threadIdx.x; j < nw; j += blockDim.x) {
    float acc = 0.f;
    const int i0 = j - c + 1 > 0 ? j - c + 1 : 0, i1 = j + c - 1 < nw - 1 ? j + c - 1 : nw - 1;
    for (int i = i0; i <= i1; ++i) acc += v[i] * M[(size_t)i * band + (j - i + c - 1)];
    out[j] = acc;
  }
}

// read-out of token r: y = B_t r W + D_t r S - ((r L^T) Mw) R  (through the
// MLP at depth 2); one block per (token, unit)
__global__ void __launch_bounds__(256) k_surp_readout(Geom g, Chunk ch, Work w, int buf, float* y) {
  extern __shared__ float sm[];
  const int u = blockIdx.y, r = blockIdx.x, t = ch.s + r;
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1;
  float* rs = sm;              // F
  float* gm = rs + g.F;        // Kw
  float* gm2 = gm + g.Kw;      // Kw
  float* aq = gm2 + g.Kw;      // hidden (depth 2)
  const float* rq = w.R + ((size_t)u * g.T + t) * g.F;
  for (int f = threadIdx.x; f < g.F; f += blockDim.x) rs[f] = rq[f];
  __syncthreads();
  const int rr = g.readout == ATLAS_READOUT_PRE ? r - 1 : r;
  const float Bt = rr < 0 ? 1.f : w.Bp[(size_t)u * g.C + rr], Dt = rr < 0 ? 0.f : w.Dp[(size_t)u * g.C + rr];
  const float* Xw = lfac(g, ch, w, u, 0);
  for (int i = threadIdx.x; i < ch.nw; i += blockDim.x) {
    float acc = 0.f;
    for (int f = 0; f < g.F; ++f) acc += rs[f] * Xw[(size_t)i * g.F + f];
    gm[i] = acc;
  }
  __syncthreads();
  const float* mwb = w.surp + (size_t)u * S.per_unit + S.mwb;
  band_mix(g, ch.nw, gm, mwb + (size_t)r * g.Kw * band, gm2);
  __syncthreads();
  float* yo = y + ((size_t)u * g.T + t) * g.d_v;
  if (g.depth == 1) {
    const float* W = w.Wst[buf][0] + (size_t)u * g.F * g.d_v;
    const float* Sb = w.Sst[buf][0] + (size_t)u * g.F * g.d_v;
    const float* DY = rfac(g, w, u, 0);
    for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
      float a = 0.f, b = 0.f, c2 = 0.f;
      for (int f = 0; f < g.F; ++f) {
        a += rs[f] * W[(size_t)f * g.d_v + k];
        b += rs[f] * Sb[(size_t)f * g.d_v + k];
      }
      for (int j = 0; j < ch.nw; ++j) c2 += gm2[j] * DY[(size_t)j * g.d_v + k];
      yo[k] = Bt * a + Dt * b - c2;
    }
    return;
  }
  const int h = g.hidden;
  const float* W1 = w.Wst[buf][0] + (size_t)u * g.F * h;
  const float* S1 = w.Sst[buf][0] + (size_t)u * g.F * h;
  const float* DZ = rfac(g, w, u, 0);
  for (int k = threadIdx.x; k < h; k += blockDim.x) {
    float a = 0.f, b = 0.f, c2 = 0.f;
    for (int f = 0; f < g.F; ++f) {
      a += rs[f] * W1[(size_t)f * h + k];
      b += rs[f] * S1[(size_t)f * h + k];
    }
    for (int j = 0; j < ch.nw; ++j) c2 += gm2[j] * DZ[(size_t)j * h + k];
    aq[k] = siluf_(Bt * a + Dt * b - c2);
  }
  __syncthreads();
  const float* Aw = lfac(g, ch, w, u, 1);
  for (int i = threadIdx.x; i < ch.nw; i += blockDim.x) {
    float acc = 0.f;
    for (int k = 0; k < h; ++k) acc += aq[k] * Aw[(size_t)i * h + k];
    gm[i] = acc;
  }
  __syncthreads();
  band_mix(g, ch.nw, gm, mwb + ((size_t)g.C + r) * g.Kw * band, gm2);
  __syncthreads();
  const float* W2 = w.Wst[buf][1] + (size_t)u * h * g.d_v;
  const float* S2 = w.Sst[buf][1] + (size_t)u * h * g.d_v;
  const float* DY = rfac(g, w, u, 1);
  for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
    float a = 0.f, b = 0.f, c2 = 0.f;
    for (int j2 = 0; j2 < h; ++j2) {
      a += aq[j2] * W2[(size_t)j2 * g.d_v + k];
      b += aq[j2] * S2[(size_t)j2 * g.d_v + k];
    }
    for (int j = 0; j < ch.nw; ++j) c2 += gm2[j] * DY[(size_t)j * g.d_v + k];
    yo[k] = rs[k] + Bt * a + Dt * b - c2;
  }
}

// Ms_e R and Mw_e R for window row i of matrix m (which = 0: Ms, 1: Mw)
__global__ void __launch_bounds__(256) k_surp_rprime(Geom g, Chunk ch, Work w) {
  const int i = blockIdx.x, m = blockIdx.y >> 1, which = blockIdx.y & 1, u = blockIdx.z;
  const SurpLayout S = surp_layout(g);
  const int band = 2 * g.c - 1, c = g.c, cols = g.cols[m], mc = max_cols(g);
  const float* base = w.surp + (size_t)u * S.per_unit;
  const float* M = base + (which ? S.mwe : S.mse) + ((size_t)m * g.Kw + i) * band;
  const float* R = rfac(g, w, u, m);
  float* out = w.surp + (size_t)u * S.per_unit + S.rp + (((size_t)m * 2 + which) * g.Kw + i) * mc;
  const int j0 = i - c + 1 > 0 ? i - c + 1 : 0, j1 = i + c - 1 < ch.nw - 1 ? i + c - 1 : ch.nw - 1;
  for (int b = threadIdx.x; b < cols; b += blockDim.x) {
    float acc = 0.f;
    for (int j = j0; j <= j1; ++j) acc += M[j - i + c - 1] * R[(size_t)j * cols + b];
    out[b] = acc;
  }
}

// chunk-end state: S = A_e Sbar - L^T (Ms_e R), W = B_e Wbar + D_e Sbar - L^T (Mw_e R)
__global__ void k_surp_state(Geom g, Chunk ch, Work w, int m, int buf) {
  const int u = blockIdx.y;
  const int rows = g.rows[m], cols = g.cols[m];
  const size_t n = (size_t)rows * cols;
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const int a = (int)(e / cols), b = (int)(e % cols);
  const SurpLayout S = surp_layout(g);
  const int mc = max_cols(g);
  const float* L = lfac(g, ch, w, u, m);
  const float* rps = w.surp + (size_t)u * S.per_unit + S.rp + ((size_t)m * 2 + 0) * g.Kw * mc;
  const float* rpw = rps + (size_t)g.Kw * mc;
  float accs = 0.f, accw = 0.f;
  for (int i = 0; i < ch.nw; ++i) {
    const float l = L[(size_t)i * rows + a];
    accs += l * rps[(size_t)i * mc + b];
    accw += l * rpw[(size_t)i * mc + b];
  }
  const int re = ch.e - 1 - ch.s;
  const float Ae = w.Ap[(size_t)u * g.C + re], Be = w.Bp[(size_t)u * g.C + re], De = w.Dp[(size_t)u * g.C + re];
  const size_t o = (size_t)u * n + e;
  const float Sb = w.Sst[buf][m][o], Wb = w.Wst[buf][m][o];
  w.Sst[buf ^ 1][m][o] = Ae * Sb - accs;
  w.Wst[buf ^ 1][m][o] = Be * Wb + De * Sb - accw;
}

}  // namespace

size_t surprise_floats(const Geom& g, size_t units) { return units * surp_layout(g).per_unit; }

cudaError_t surprise_chunk(const Geom& g, const Chunk& ch, const Work& w, const float* theta, const float* eta,
                           const float* alpha, float* y, int buf, cudaStream_t st, int* nl) {
  const int Ct = ch.e - ch.s, band = 2 * g.c - 1;
  k_surp_gram<<<dim3(ch.nw, g.nmat * 2, g.units), 256, 0, st>>>(g, ch, w);
  k_surp_ns<<<dim3(Ct, g.nmat, g.units), 256, 0, st>>>(g, ch, w);
  k_surp_scan<<<dim3((g.Kw * band + 255) / 256, g.nmat, g.units), 256, 0, st>>>(g, ch, w, theta, eta, alpha);
  const size_t sr = (size_t)(g.F + 2 * g.Kw + (g.depth == 2 ? g.hidden : 0)) * sizeof(float);
  cudaFuncSetAttribute(k_surp_readout, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sr);
  k_surp_readout<<<dim3(Ct, g.units), 256, sr, st>>>(g, ch, w, buf, y);
  k_surp_rprime<<<dim3(ch.nw, g.nmat * 2, g.units), 256, 0, st>>>(g, ch, w);
  for (int m = 0; m < g.nmat; ++m) {
    const size_t n = (size_t)g.rows[m] * g.cols[m];
    k_surp_state<<<dim3((unsigned)((n + 255) / 256), g.units), 256, 0, st>>>(g, ch, w, m, buf);
  }
  *nl += 5 + g.nmat;
  return cudaGetLastError();
}

}  // namespace atlas
