// Generic fp32 SIMT kernels of the chunked memory forward.
//
// These cover every configuration the API accepts (any depth, widths, chunk,
// window, feature map and Newton-Schulz count within the limits checked on
// the host) in plain fp32 arithmetic.  The per-chunk work is split into small
// kernels launched in order on one stream:
//
//   grad     gradient factors of the window rows at the chunk-start weights
//   coef     gate scans: coefficients of every window row in S_t and W_t
//   dual_*   (no Newton-Schulz) read-out and chunk-end state in dual form
//   ns_*     (Newton-Schulz) per-token momentum, orthogonalisation, decay
//            scan and read-out
//
// Notation (row vectors): window row i is key token lo+i of the chunk;
// x_i its features, a_i = SiLU(z_i), z_i = x_i W1bar; dy_i = 2 gamma_i
// (M_Wbar(x_i) - v_i); dz_i = (dy_i W2bar^T) * SiLU'(z_i).  Then
//   S_t = A_t Sbar - sum_i Cs[t,i] G_i,   W_t = B_t Wbar + D_t Sbar - sum_i Cw[t,i] G_i
// with G_i the per-token gradient outer products (x_i^T dy_i at depth 1;
// x_i^T dz_i and a_i^T dy_i at depth 2), A_t = prod eta, B_t = prod (1-alpha),
// Cs[t,i] = eta_t Cs[t-1,i] + theta_t [i in window(t)], Cw[t,i] = (1-alpha_t)
// Cw[t-1,i] + Cs[t,i], D_t = (1-alpha_t) D_{t-1} + A_t: the Titans recurrences
// (titans-pytorch-mlx README, Eq. 13-14) unrolled over one chunk whose
// gradients are all taken at the chunk-start weights (ATLAS summary, 3.3).
#include "atlas_common.cuh"
#include "simt_tile.cuh"

namespace atlas {

// ------------------------------------------------------------------ features
// phi(x): identity, or [1, x_i, x_i x_j / 2 (i <= j, lexicographic)], then
// optionally times P (atlas-torch README, "Atlas Extensions": Polynomial
// Features).  One block per token row.
__device__ __forceinline__ float poly_feature(const float* x, int d, int f) {
  if (f == 0) return 1.f;
  if (f <= d) return x[f - 1];
  int q = f - 1 - d, i = 0;
  while (q >= d - i) { q -= d - i; ++i; }
  return 0.5f * x[i] * x[i + q];
}

__global__ void k_features(Geom g, const void* src, const void* cache, int rows_per_unit,
                           int from_cache, const void* P, float* out) {
  extern __shared__ float sm[];
  float* x = sm;             // d_k
  float* phi = sm + g.d_k;   // poly (only when projecting)
  const int u = blockIdx.y, row = blockIdx.x;
  const int d = g.d_k;
  // where does this row come from: the window cache or the call's tokens
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    float val;
    if (from_cache && row < g.n_prev) {
      size_t slot = (size_t)(g.c - 1 - g.n_prev + row);
      val = load_in(cache, ((size_t)u * (g.c - 1) + slot) * d + k, g.qkv_dtype);
    } else {
      int t = row - (from_cache ? g.n_prev : 0);
      val = load_in(src, ((size_t)u * g.T + t) * d + k, g.qkv_dtype);
    }
    x[k] = val;
  }
  __syncthreads();
  float* o = out + ((size_t)u * rows_per_unit + row) * g.F;
  if (g.proj_dim == 0) {
    for (int f = threadIdx.x; f < g.F; f += blockDim.x) o[f] = g.p == 1 ? x[f] : poly_feature(x, d, f);
    return;
  }
  for (int f = threadIdx.x; f < g.poly; f += blockDim.x) phi[f] = g.p == 1 ? x[f] : poly_feature(x, d, f);
  __syncthreads();
  for (int j = threadIdx.x; j < g.proj_dim; j += blockDim.x) {
    float acc = 0.f;
    for (int f = 0; f < g.poly; ++f) acc += phi[f] * load_in(P, (size_t)f * g.proj_dim + j, g.qkv_dtype);
    o[j] = acc;
  }
}

// values and Omega weights of every key row (cache rows first)
__global__ void k_values(Geom g, const void* v, const void* win_v, const float* gamma,
                         const float* win_gamma, float* V, float* G) {
  const int u = blockIdx.y, row = blockIdx.x;
  const bool cached = row < g.n_prev;
  const size_t slot = (size_t)(g.c - 1 - g.n_prev + row);
  const int t = row - g.n_prev;
  for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
    float val = cached ? load_in(win_v, ((size_t)u * (g.c - 1) + slot) * g.d_v + k, g.qkv_dtype)
                       : load_in(v, ((size_t)u * g.T + t) * g.d_v + k, g.qkv_dtype);
    V[((size_t)u * g.L + row) * g.d_v + k] = val;
  }
  if (threadIdx.x == 0) {
    float gm = 1.f;
    if (cached) { if (win_gamma) gm = win_gamma[(size_t)u * (g.c - 1) + slot]; }
    else if (gamma) gm = gamma[(size_t)u * g.T + t];
    G[(size_t)u * g.L + row] = gm;
  }
}


// --------------------------------------------------------------------- coef
// One block per unit, one thread per window row (plus thread 0 for the
// per-token products).  Sequential over the tokens of the chunk.
__global__ void k_coef(Geom g, Chunk ch, const float* theta, const float* eta, const float* alpha, Work w) {
  // the chunk's gates in shared memory first: the scans below then run
  // without a global-memory round trip per token
  extern __shared__ float gates[];   // [3][C]: theta, eta, 1 - alpha
  const int u = blockIdx.x;
  const int i = threadIdx.x;
  const int Ct = ch.e - ch.s;
  for (int r = threadIdx.x; r < Ct; r += blockDim.x) {
    gates[r] = theta[(size_t)u * g.T + ch.s + r];
    gates[g.C + r] = eta[(size_t)u * g.T + ch.s + r];
    gates[2 * g.C + r] = 1.f - alpha[(size_t)u * g.T + ch.s + r];
  }
  __syncthreads();
  const int ti = ch.lo + i;  // token index of window row i (may be < 0: cached)
  float cs = 0.f, cw = 0.f, Ap = 1.f, Bp = 1.f, Dp = 0.f;
  for (int r = 0; r < Ct; ++r) {
    const int t = ch.s + r;
    const float th = gates[r], et = gates[g.C + r], be = gates[2 * g.C + r];
    if (i < ch.nw) {
      const bool in_win = ti <= t && t <= ti + g.c - 1;
      cs = et * cs + (in_win ? th : 0.f);
      cw = be * cw + cs;
      w.Cs[((size_t)u * g.C + r) * g.Kw + i] = cs;
      w.Cw[((size_t)u * g.C + r) * g.Kw + i] = cw;
    }
    if (i == 0) {
      Ap *= et;
      Bp *= be;
      Dp = be * Dp + Ap;
      w.Ap[(size_t)u * g.C + r] = Ap;
      w.Bp[(size_t)u * g.C + r] = Bp;
      w.Dp[(size_t)u * g.C + r] = Dp;
    }
  }
}

// Chunk-wise update rule (titans-pytorch store path, as the atlas-torch
// README's per_token_updates fix describes it): the same coefficient arrays
// for a memory that changes once per chunk.  With c = 1 window row i is
// token s + i.  Before the chunk's last token nothing has changed: S_t is
// reported as 0 (Newton-Schulz, if any, is skipped there and adds U = 0), W_t
// = W_bar.  At the last token S_e = eta_bar S_bar - sum_i theta_i g_i and
// W_e = (1 - alpha_bar) W_bar + eta_bar S_bar - sum_i theta_i g_i, with
// eta_bar, alpha_bar the chunk's mean gates.  One block per unit.
__global__ void k_coef_chunkwise(Geom g, Chunk ch, const float* theta, const float* eta, const float* alpha,
                                 Work w) {
  __shared__ float red[2][32];
  const int u = blockIdx.x;
  const int Ct = ch.e - ch.s;
  const size_t base = (size_t)u * g.T + ch.s;
  float se = 0.f, sa = 0.f;
  for (int r = threadIdx.x; r < Ct; r += blockDim.x) {
    se += eta[base + r];
    sa += alpha[base + r];
  }
  for (int o = 16; o > 0; o >>= 1) {
    se += __shfl_xor_sync(0xffffffffu, se, o);
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
  }
  if (threadIdx.x % 32 == 0) {
    red[0][threadIdx.x / 32] = se;
    red[1][threadIdx.x / 32] = sa;
  }
  __syncthreads();
  se = sa = 0.f;
  for (int k = 0; k < (int)(blockDim.x / 32); ++k) {
    se += red[0][k];
    sa += red[1][k];
  }
  const float eb = se / Ct, ab = sa / Ct;
  for (int e = threadIdx.x; e < Ct * ch.nw; e += blockDim.x) {
    const int r = e / ch.nw, i = e % ch.nw;
    const float v = r == Ct - 1 ? theta[base + i] : 0.f;
    w.Cs[((size_t)u * g.C + r) * g.Kw + i] = v;
    w.Cw[((size_t)u * g.C + r) * g.Kw + i] = v;
  }
  for (int r = threadIdx.x; r < Ct; r += blockDim.x) {
    const bool last = r == Ct - 1;
    w.Ap[(size_t)u * g.C + r] = last ? eb : 0.f;
    w.Bp[(size_t)u * g.C + r] = last ? 1.f - ab : 1.f;
    w.Dp[(size_t)u * g.C + r] = last ? eb : 0.f;
    if (w.aeff) w.aeff[base + r] = last ? ab : 0.f;   // the decay the W scans apply
  }
}

// ---------------------------------------------------------------- dual form
// Read-out without Newton-Schulz.  One block per (token of chunk, unit).
__global__ void k_dual_readout(Geom g, Chunk ch, Work w, int buf, float* y) {
  extern __shared__ float sm[];
  const int u = blockIdx.y, r = blockIdx.x, t = ch.s + r;
  float* rs = sm;                  // F
  float* gm = rs + g.F;            // nw  (r . x_i, later aq . a_i)
  float* cw = gm + g.Kw;           // nw
  const float* rq = w.R + ((size_t)u * g.T + t) * g.F;
  for (int f = threadIdx.x; f < g.F; f += blockDim.x) rs[f] = rq[f];
  // read-out coefficients: token r's own, or in pre-update mode token
  // r - 1's (the chunk-start state for r = 0: Cw = 0, B = 1, D = 0)
  const int rr = g.readout == ATLAS_READOUT_PRE ? r - 1 : r;
  for (int i = threadIdx.x; i < ch.nw; i += blockDim.x) cw[i] = rr < 0 ? 0.f : w.Cw[((size_t)u * g.C + rr) * g.Kw + i];
  __syncthreads();
  const float Bt = rr < 0 ? 1.f : w.Bp[(size_t)u * g.C + rr], Dt = rr < 0 ? 0.f : w.Dp[(size_t)u * g.C + rr];
  const float* Xw = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
  for (int i = threadIdx.x; i < ch.nw; i += blockDim.x) {
    float acc = 0.f;
    for (int f = 0; f < g.F; ++f) acc += rs[f] * Xw[(size_t)i * g.F + f];
    gm[i] = acc * cw[i];
  }
  __syncthreads();
  float* yo = y + ((size_t)u * g.T + t) * g.d_v;
  if (g.depth == 1) {
    const float* W = w.Wst[buf][0] + (size_t)u * g.F * g.d_v;
    const float* S = w.Sst[buf][0] + (size_t)u * g.F * g.d_v;
    for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
      float a = 0.f, b = 0.f, c = 0.f;
      for (int f = 0; f < g.F; ++f) {
        a += rs[f] * W[(size_t)f * g.d_v + k];
        b += rs[f] * S[(size_t)f * g.d_v + k];
      }
      for (int i = 0; i < ch.nw; ++i) c += gm[i] * w.DY[((size_t)u * g.Kw + i) * g.d_v + k];
      yo[k] = Bt * a + Dt * b - c;
    }
    return;
  }
  const int h = g.hidden;
  float* aq = cw + g.Kw;          // h
  const float* W1 = w.Wst[buf][0] + (size_t)u * g.F * h;
  const float* S1 = w.Sst[buf][0] + (size_t)u * g.F * h;
  for (int j = threadIdx.x; j < h; j += blockDim.x) {
    float a = 0.f, b = 0.f, c = 0.f;
    for (int f = 0; f < g.F; ++f) {
      a += rs[f] * W1[(size_t)f * h + j];
      b += rs[f] * S1[(size_t)f * h + j];
    }
    for (int i = 0; i < ch.nw; ++i) c += gm[i] * w.DZ[((size_t)u * g.Kw + i) * h + j];
    aq[j] = siluf_(Bt * a + Dt * b - c);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ch.nw; i += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < h; ++j) acc += aq[j] * w.Aact[((size_t)u * g.Kw + i) * h + j];
    gm[i] = acc * cw[i];
  }
  __syncthreads();
  const float* W2 = w.Wst[buf][1] + (size_t)u * h * g.d_v;
  const float* S2 = w.Sst[buf][1] + (size_t)u * h * g.d_v;
  for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
    float a = 0.f, b = 0.f, c = 0.f;
    for (int j = 0; j < h; ++j) {
      a += aq[j] * W2[(size_t)j * g.d_v + k];
      b += aq[j] * S2[(size_t)j * g.d_v + k];
    }
    for (int i = 0; i < ch.nw; ++i) c += gm[i] * w.DY[((size_t)u * g.Kw + i) * g.d_v + k];
    yo[k] = rs[k] + Bt * a + Dt * b - c;
  }
}

// left/right factors of window row i for matrix m
__device__ __forceinline__ const float* left_factor(const Geom& g, const Chunk& ch, const Work& w, int u, int m) {
  if (g.depth == 2 && m == 1) return w.Aact + (size_t)u * g.Kw * g.hidden;
  return w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
}
__device__ __forceinline__ const float* right_factor(const Geom& g, const Work& w, int u, int m) {
  if (g.depth == 2 && m == 0) return w.DZ + (size_t)u * g.Kw * g.hidden;
  return w.DY + (size_t)u * g.Kw * g.d_v;
}

// Chunk-end state without Newton-Schulz; one thread per matrix element.
__global__ void k_dual_state(Geom g, Chunk ch, Work w, int m, int buf) {
  const int u = blockIdx.y;
  const int rows = g.rows[m], cols = g.cols[m];
  const size_t n = (size_t)rows * cols;
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const int a = (int)(e / cols), b = (int)(e % cols);
  const float* Lf = left_factor(g, ch, w, u, m);
  const float* Rf = right_factor(g, w, u, m);
  const int r = ch.e - 1 - ch.s;
  const float* cs = w.Cs + ((size_t)u * g.C + r) * g.Kw;
  const float* cwv = w.Cw + ((size_t)u * g.C + r) * g.Kw;
  float accs = 0.f, accw = 0.f;
  for (int i = 0; i < ch.nw; ++i) {
    const float prod = Lf[(size_t)i * rows + a] * Rf[(size_t)i * cols + b];
    accs += cs[i] * prod;
    accw += cwv[i] * prod;
  }
  const float Ae = w.Ap[(size_t)u * g.C + r], Be = w.Bp[(size_t)u * g.C + r], De = w.Dp[(size_t)u * g.C + r];
  const size_t o = (size_t)u * n + e;
  const float Sb = w.Sst[buf][m][o], Wb = w.Wst[buf][m][o];
  w.Sst[buf ^ 1][m][o] = Ae * Sb - accs;
  w.Wst[buf ^ 1][m][o] = Be * Wb + De * Sb - accw;
}

// ------------------------------------------------------------ Newton-Schulz

// One block per (token from ns_first_row on, matrix, unit): form S_t,
// orthogonalise, store U_t in the token's slot of Ubuf (X orientation: the
// short side first).
// Shared memory: Am[rX*rX] + Bm[rX*rX] + 2 tiles of 16x64.
__global__ void __launch_bounds__(256) k_ns_simt(Geom g, Chunk ch, Work w, int buf, int m, size_t slot_stride,
                                                  size_t slot_off) {
  extern __shared__ float sm[];
  const int u = blockIdx.y, r = ns_first_row(g, ch) + blockIdx.x, t = ch.s + r;
  const int rows = g.rows[m], cols = g.cols[m];
  const bool tall = rows > cols;
  const int rX = tall ? cols : rows, cX = tall ? rows : cols;
  float* Am = sm;
  float* Bm = sm + rX * rX;
  float* As = Bm + rX * rX;
  float* Bs = As + 16 * 64;
  __shared__ float red[32];
  float* X = w.Ubuf + ((size_t)u * g.C + r) * slot_stride + slot_off;
  const size_t n = (size_t)rows * cols;
  const float* Lf = left_factor(g, ch, w, u, m);
  const float* Rf = right_factor(g, w, u, m);
  const float* cs = w.Cs + ((size_t)u * g.C + r) * g.Kw;
  const float At = w.Ap[(size_t)u * g.C + r];
  const float* Sb = w.Sst[buf][m] + (size_t)u * n;
  const bool last = (t == ch.e - 1);
  float ss = 0.f;
  for (size_t e = threadIdx.x; e < n; e += blockDim.x) {
    const int a = (int)(e / cols), b = (int)(e % cols);
    float acc = 0.f;
    for (int i = 0; i < ch.nw; ++i) acc += cs[i] * Lf[(size_t)i * rows + a] * Rf[(size_t)i * cols + b];
    const float val = At * Sb[e] - acc;
    if (last) w.Sst[buf ^ 1][m][(size_t)u * n + e] = val;
    X[tall ? (size_t)b * cX + a : e] = val;
    ss += val * val;
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int k = 0; k < (int)(blockDim.x / 32); ++k) tot += red[k];
    red[0] = 1.f / (sqrtf(tot) + kNsEps);
  }
  __syncthreads();
  const float scale = red[0];
  for (size_t e = threadIdx.x; e < n; e += blockDim.x) X[e] *= scale;
  __syncthreads();
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int it = 0; it < g.ns_iters; ++it) {
    // A = X X^T
    for (int i0 = 0; i0 < rX; i0 += 64)
      for (int j0 = 0; j0 < rX; j0 += 64) {
        float acc[4][4];
        tile_gemm(TileOp{X, cX, 1}, TileOp{X, cX, 1}, rX, rX, cX, i0, j0, acc, As, Bs);
        for (int a = 0; a < 4; ++a)
          for (int b = 0; b < 4; ++b) {
            const int i = i0 + ty * 4 + a, j = j0 + tx * 4 + b;
            if (i < rX && j < rX) Am[i * rX + j] = acc[a][b];
          }
      }
    __syncthreads();
    // B = a I + b A + c A A
    for (int i0 = 0; i0 < rX; i0 += 64)
      for (int j0 = 0; j0 < rX; j0 += 64) {
        float acc[4][4];
        tile_gemm(TileOp{Am, rX, 1}, TileOp{Am, 1, rX}, rX, rX, rX, i0, j0, acc, As, Bs);
        for (int a = 0; a < 4; ++a)
          for (int b = 0; b < 4; ++b) {
            const int i = i0 + ty * 4 + a, j = j0 + tx * 4 + b;
            if (i < rX && j < rX) Bm[i * rX + j] = kNsB * Am[i * rX + j] + kNsC * acc[a][b] + (i == j ? kNsA : 0.f);
          }
      }
    __syncthreads();
    // X <- B X, one column block at a time (a column block only reads itself)
    for (int j0 = 0; j0 < cX; j0 += 64) {
      float keep[2][4][4];
      for (int ib = 0; ib < (rX + 63) / 64; ++ib) {
        float acc[4][4];
        tile_gemm(TileOp{Bm, rX, 1}, TileOp{X, 1, cX}, rX, cX, rX, ib * 64, j0, acc, As, Bs);
        // rX <= 128 (checked on the host): at most two row blocks
        for (int a = 0; a < 4; ++a)
          for (int b = 0; b < 4; ++b) keep[ib & 1][a][b] = acc[a][b];
      }
      __syncthreads();
      for (int ib = 0; ib < (rX + 63) / 64; ++ib)
        for (int a = 0; a < 4; ++a)
          for (int b = 0; b < 4; ++b) {
            const int i = ib * 64 + ty * 4 + a, j = j0 + tx * 4 + b;
            if (i < rX && j < cX) X[(size_t)i * cX + j] = keep[ib & 1][a][b];
          }
      __syncthreads();
    }
  }
}

// Decay scan over the chunk, in place: slot t holds U_t on entry and the
// weights token t reads out on exit: W_t, or W_{t-1} in pre-update mode
// (W_{s-1} = Wbar).  One thread per matrix element (X orientation).
__global__ void k_ns_wscan(Geom g, Chunk ch, Work w, int buf, int m, size_t slot_stride, size_t slot_off,
                           const float* alpha) {
  const int u = blockIdx.y;
  const int rows = g.rows[m], cols = g.cols[m];
  const bool tall = rows > cols;
  const size_t n = (size_t)rows * cols;
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const int a = (int)(e / cols), b = (int)(e % cols);
  const size_t xe = tall ? (size_t)b * rows + a : e;
  float W = w.Wst[buf][m][(size_t)u * n + e];
  const bool pre = g.readout == ATLAS_READOUT_PRE;
  const int rn = ns_first_row(g, ch);   // slots before it hold no U_t: U_t = 0
  for (int t = ch.s; t < ch.e; ++t) {
    float* slot = w.Ubuf + ((size_t)u * g.C + (t - ch.s)) * slot_stride + slot_off;
    const float W_prev = W;
    W = (1.f - alpha[(size_t)u * g.T + t]) * W + (t - ch.s >= rn ? slot[xe] : 0.f);
    slot[xe] = pre ? W_prev : W;   // the weights token t reads out
  }
  w.Wst[buf ^ 1][m][(size_t)u * n + e] = W;
}

// Read-out from the materialised per-token weights W_t (Newton-Schulz path).
__global__ void k_ns_readout(Geom g, Chunk ch, Work w, size_t slot_stride, float* y) {
  extern __shared__ float sm[];
  const int u = blockIdx.y, r = blockIdx.x, t = ch.s + r;
  float* rs = sm;
  const float* rq = w.R + ((size_t)u * g.T + t) * g.F;
  for (int f = threadIdx.x; f < g.F; f += blockDim.x) rs[f] = rq[f];
  __syncthreads();
  const float* slot = w.Ubuf + ((size_t)u * g.C + r) * slot_stride;
  float* yo = y + ((size_t)u * g.T + t) * g.d_v;
  if (g.depth == 1) {
    const bool tall = g.F > g.d_v;
    for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
      float acc = 0.f;
      for (int f = 0; f < g.F; ++f) acc += rs[f] * slot[tall ? (size_t)k * g.F + f : (size_t)f * g.d_v + k];
      yo[k] = acc;
    }
    return;
  }
  const int h = g.hidden;
  float* aq = rs + g.F;
  const bool tall1 = g.F > h;
  for (int j = threadIdx.x; j < h; j += blockDim.x) {
    float acc = 0.f;
    for (int f = 0; f < g.F; ++f) acc += rs[f] * slot[tall1 ? (size_t)j * g.F + f : (size_t)f * h + j];
    aq[j] = siluf_(acc);
  }
  __syncthreads();
  const float* W2 = slot + (size_t)g.F * h;
  const bool tall2 = h > g.d_v;
  for (int k = threadIdx.x; k < g.d_v; k += blockDim.x) {
    float acc = rs[k];
    for (int j = 0; j < h; ++j) acc += aq[j] * W2[tall2 ? (size_t)k * h + j : (size_t)j * g.d_v + k];
    yo[k] = acc;
  }
}

// Outgoing window cache: gather the last c-1 raw tokens into a temporary.
__global__ void k_cache_gather(Geom g, const void* k, const void* v, const float* gamma, const void* win_k,
                               const void* win_v, const float* win_gamma, float* tmp) {
  const int u = blockIdx.y, slot = blockIdx.x;  // slot in [0, c-1)
  const int total = g.n_prev + g.T;
  const int j = total - (g.c - 1) + slot;       // key row; < 0 means empty
  const int width = g.d_k + g.d_v + 1;
  float* o = tmp + ((size_t)u * (g.c - 1) + slot) * width;
  if (j < 0) return;
  const bool cached = j < g.n_prev;
  const size_t cs = (size_t)u * (g.c - 1) + (g.c - 1 - g.n_prev + j);
  const size_t ts = (size_t)u * g.T + (j - g.n_prev);
  for (int e = threadIdx.x; e < width; e += blockDim.x) {
    float val;
    if (e < g.d_k) val = cached ? load_in(win_k, cs * g.d_k + e, g.qkv_dtype) : load_in(k, ts * g.d_k + e, g.qkv_dtype);
    else if (e < g.d_k + g.d_v) {
      const int f = e - g.d_k;
      val = cached ? load_in(win_v, cs * g.d_v + f, g.qkv_dtype) : load_in(v, ts * g.d_v + f, g.qkv_dtype);
    } else {
      val = cached ? (win_gamma ? win_gamma[cs] : 1.f) : (gamma ? gamma[ts] : 1.f);
    }
    o[e] = val;
  }
}

__device__ __forceinline__ void store_out(void* p, size_t i, float val, int dtype) {
  if (dtype == ATLAS_BF16) {
    // the gathered values are exact copies of bf16 inputs: truncation is exact
    ((uint16_t*)p)[i] = (uint16_t)(__float_as_uint(val) >> 16);
  } else {
    ((float*)p)[i] = val;
  }
}

__global__ void k_cache_scatter(Geom g, const float* tmp, void* k_out, void* v_out, float* g_out) {
  const int u = blockIdx.y, slot = blockIdx.x;
  const int total = g.n_prev + g.T;
  const int j = total - (g.c - 1) + slot;
  if (j < 0) return;
  const int width = g.d_k + g.d_v + 1;
  const float* s = tmp + ((size_t)u * (g.c - 1) + slot) * width;
  const size_t cs = (size_t)u * (g.c - 1) + slot;
  for (int e = threadIdx.x; e < width; e += blockDim.x) {
    if (e < g.d_k) { if (k_out) store_out(k_out, cs * g.d_k + e, s[e], g.qkv_dtype); }
    else if (e < g.d_k + g.d_v) { if (v_out) store_out(v_out, cs * g.d_v + (e - g.d_k), s[e], g.qkv_dtype); }
    else if (g_out) g_out[cs] = s[e];
  }
}

// ------------------------------------------------------------------ driver
static inline unsigned cdiv(size_t a, size_t b) { return (unsigned)((a + b - 1) / b); }

#define CUDA_CHECK_RET(x)            \
  do {                               \
    cudaError_t e_ = (x);            \
    if (e_ != cudaSuccess) return e_; \
  } while (0)

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

size_t features_proj_smem(const Geom& g);
bool features_proj_supported(const Geom& g);
cudaError_t features_proj_launch(const Geom& g, const void* src, const void* cache, int rows, int from_cache,
                                 const void* P, float* out, cudaStream_t st);

cudaError_t generic_prepare(const Geom& g, const Work& w, const GenericIO& io, cudaStream_t st, int* nl) {
  *nl += 3;
  if (features_tc_supported(g) && w.Pt) {
    // tensor cores: P transposed once, then phi(k) P and phi(q) P
    *nl += 1;
    CUDA_CHECK_RET(features_tc_prepare(g, io.P, w.Pt, st));
    CUDA_CHECK_RET(features_tc_launch(g, io.k, io.win_k, g.L, 1, w.Pt, w.X, w.status, st));
    CUDA_CHECK_RET(features_tc_launch(g, io.q, nullptr, g.T, 0, w.Pt, w.R, w.status, st));
    k_values<<<dim3(g.L, g.units), 128, 0, st>>>(g, io.v, io.win_v, io.gamma, io.win_gamma, w.V, w.G);
    return cudaGetLastError();
  }
  if (features_proj_supported(g)) {
    CUDA_CHECK_RET(features_proj_launch(g, io.k, io.win_k, g.L, 1, io.P, w.X, st));
    CUDA_CHECK_RET(features_proj_launch(g, io.q, nullptr, g.T, 0, io.P, w.R, st));
    k_values<<<dim3(g.L, g.units), 128, 0, st>>>(g, io.v, io.win_v, io.gamma, io.win_gamma, w.V, w.G);
    return cudaGetLastError();
  }
  const size_t sm_feat = (size_t)(g.d_k + (g.proj_dim ? g.poly : 0)) * sizeof(float);
  if (sm_feat > 48 * 1024) cudaFuncSetAttribute(k_features, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_feat);
  k_features<<<dim3(g.L, g.units), 128, sm_feat, st>>>(g, io.k, io.win_k, g.L, 1, io.P, w.X);
  k_features<<<dim3(g.T, g.units), 128, sm_feat, st>>>(g, io.q, nullptr, g.T, 0, io.P, w.R);
  k_values<<<dim3(g.L, g.units), 128, 0, st>>>(g, io.v, io.win_v, io.gamma, io.win_gamma, w.V, w.G);
  return cudaGetLastError();
}

// Shared-memory bytes each generic kernel needs (checked against the device
// limit on the host before launching).
size_t generic_smem_readout(const Geom& g) {
  return (size_t)(g.F + 2 * g.Kw + (g.depth == 2 ? g.hidden : 0)) * sizeof(float);
}
size_t generic_smem_ns(const Geom& g, int m) {
  const int rX = g.rows[m] < g.cols[m] ? g.rows[m] : g.cols[m];
  return (size_t)(2 * rX * rX + 2 * 16 * 64) * sizeof(float);
}

cudaError_t grad_tiled(const Geom& g, const Chunk& ch, const Work& w, int buf, cudaStream_t st, int* nl);
bool dual1_split_supported(const Geom& g);
cudaError_t dual1_split(const Geom& g, const Chunk& ch, const Work& w, const GenericIO& io, int buf,
                        cudaStream_t st, int* nl);
bool ns_fused_scan_supported(const Geom& g);
cudaError_t ns_fused_scan(const Geom& g, const Chunk& ch, const Work& w, int buf, size_t slot_stride,
                          const float* alpha, float* aq, float* y, cudaStream_t st);


cudaError_t generic_chunk(const Geom& g, const Chunk& ch, const Work& w, const GenericIO& io, int buf,
                          cudaStream_t st, int* nl) {
  if (dual1_split_supported(g)) return dual1_split(g, ch, w, io, buf, st, nl);
  if (g.ns_iters > 0 && g.ns_target == ATLAS_NS_SURPRISE) {
    CUDA_CHECK_RET(grad_tiled(g, ch, w, buf, st, nl));
    const int coef_threads = ((ch.nw + 31) / 32) * 32;
    k_coef<<<g.units, coef_threads, 3 * g.C * sizeof(float), st>>>(g, ch, io.theta, io.eta, io.alpha, w);
    *nl += 2;
    return surprise_chunk(g, ch, w, io.theta, io.eta, io.alpha, io.y, buf, st, nl);
  }
  *nl += g.ns_iters == 0 ? 3 + g.nmat : 3 + 2 * g.nmat;
  const size_t sr = generic_smem_readout(g);
  CUDA_CHECK_RET(grad_tiled(g, ch, w, buf, st, nl));
  const bool chunkwise = g.update == ATLAS_UPDATE_CHUNKWISE;
  if (chunkwise) {
    k_coef_chunkwise<<<g.units, 256, 0, st>>>(g, ch, io.theta, io.eta, io.alpha, w);
  } else {
    const int coef_threads = ((ch.nw + 31) / 32) * 32;
    k_coef<<<g.units, coef_threads, 3 * g.C * sizeof(float), st>>>(g, ch, io.theta, io.eta, io.alpha, w);
  }
  // the decay the W scans apply per token (chunk-wise: only at the chunk's end)
  const float* alpha_scan = chunkwise ? w.aeff : io.alpha;
  if (g.ns_iters == 0) {
    cudaFuncSetAttribute(k_dual_readout, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sr);
    k_dual_readout<<<dim3(ch.e - ch.s, g.units), 256, sr, st>>>(g, ch, w, buf, io.y);
    for (int m = 0; m < g.nmat; ++m) {
      const size_t n = (size_t)g.rows[m] * g.cols[m];
      k_dual_state<<<dim3(cdiv(n, 256), g.units), 256, 0, st>>>(g, ch, w, m, buf);
    }
    return cudaGetLastError();
  }
  size_t slot_stride = 0;
  for (int m = 0; m < g.nmat; ++m) slot_stride += (size_t)g.rows[m] * g.cols[m];
  size_t off = 0;
  if (ns_tc_supported(g)) {
    CUDA_CHECK_RET(ns_tc_launch(g, ch, w, buf, slot_stride, num_sms(), io.theta, io.eta, st));
    *nl -= g.nmat - 1;   // one tensor-core launch covers every matrix
  } else
  for (int m = 0; m < g.nmat; ++m) {
    const size_t sn = generic_smem_ns(g, m);
    cudaFuncSetAttribute(k_ns_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sn);
    k_ns_simt<<<dim3(ch.e - ch.s - ns_first_row(g, ch), g.units), 256, sn, st>>>(g, ch, w, buf, m, slot_stride,
                                                                                   off);
    off += (size_t)g.rows[m] * g.cols[m];
  }
  if (ns_fused_scan_supported(g)) {
    *nl -= 1;   // two fused launches replace nmat scans + one read-out
    return ns_fused_scan(g, ch, w, buf, slot_stride, alpha_scan, w.Zpre, io.y, st);
  }
  off = 0;
  for (int m = 0; m < g.nmat; ++m) {
    const size_t n = (size_t)g.rows[m] * g.cols[m];
    k_ns_wscan<<<dim3(cdiv(n, 256), g.units), 256, 0, st>>>(g, ch, w, buf, m, slot_stride, off, alpha_scan);
    off += n;
  }
  const size_t srd = (size_t)(g.F + (g.depth == 2 ? g.hidden : 0)) * sizeof(float);
  cudaFuncSetAttribute(k_ns_readout, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)srd);
  k_ns_readout<<<dim3(ch.e - ch.s, g.units), 256, srd, st>>>(g, ch, w, slot_stride, io.y);
  return cudaGetLastError();
}

cudaError_t generic_cache_out(const Geom& g, const GenericIO& io, float* tmp, void* k_out, void* v_out,
                              float* g_out, cudaStream_t st, int* nl) {
  if (g.c <= 1) return cudaSuccess;
  *nl += 2;
  k_cache_gather<<<dim3(g.c - 1, g.units), 128, 0, st>>>(g, io.k, io.v, io.gamma, io.win_k, io.win_v, io.win_gamma,
                                                         tmp);
  k_cache_scatter<<<dim3(g.c - 1, g.units), 128, 0, st>>>(g, tmp, k_out, v_out, g_out);
  return cudaGetLastError();
}

}  // namespace atlas

namespace atlas {

// Asynchronous 4-byte global -> shared copies: every load of a stage is in
// flight at once instead of one round trip per loop iteration.  An invalid
// element copies 0 bytes from a valid address and zero-fills.
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool valid, const float* fallback) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(valid ? src : fallback),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// 16-byte copy (both addresses 16-byte aligned)
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// --------------------------------------------- fused decay scan + read-out
// Newton-Schulz path, depth 2 with W1 (F x h, F <= h) and W2 (h x d, h > d),
// both stored per token in Ubuf in the X orientation (W1 as is, W2
// transposed).  W_t = (1 - alpha_t) W_{t-1} + U_t is scanned in registers;
// every U_t is read once and no W_t is written back, only W_e.
//
// Pass 1: z_t = r_t W1_t, aq_t = SiLU(z_t).  CTA = (unit, 32 columns of W1);
// thread = (column j = lane, row group g = warp): rows [g * rpg, (g+1) * rpg)
// in registers; partial dot products meet in shared memory.
template <int RPG>
__global__ void __launch_bounds__(256) k_ns_scan_w1(Geom g, Chunk ch, Work w, int buf, size_t slot_stride,
                                                    const float* alpha, float* aq) {
  // W1 decay scan fused with the hidden read-out.  Thread (grp, lane) keeps
  // rows [grp RPG, grp RPG + RPG) of column jb + lane of W1.  The U_t of
  // PD tokens are loaded together; each token's partial dot products go to
  // shared memory and are summed over the 8 row groups once at the end, so
  // the token loop has no barrier.  PD RPG = 64 values in flight per thread.
  constexpr int PD = 64 / RPG;
  extern __shared__ float scan_sm[];
  const int u = blockIdx.y, jb = blockIdx.x * 32;
  const int lane = threadIdx.x % 32, grp = threadIdx.x / 32;
  const int F = g.F, h = g.hidden, j = jb + lane, i0 = grp * RPG;
  const int Ct = ch.e - ch.s;
  const bool pre = g.readout == ATLAS_READOUT_PRE;   // read out before token r's update
  const int rn = ns_first_row(g, ch);                 // slots before it hold no U_t: U_t = 0
  float* rq = scan_sm;                   // [C][F + 1] queries of the chunk
  float* part = rq + g.C * (F + 1);      // [C][8][33] per-group partial sums
  float* bes = part + g.C * 8 * 33;      // [C] 1 - alpha
  // the chunk's queries by cp.async (all in flight at once), then the gates
  for (int e = threadIdx.x; e < Ct * F; e += 256)
    cp_async4(&rq[(e / F) * (F + 1) + e % F], &w.R[((size_t)u * g.T + ch.s + e / F) * F + e % F], true, w.R);
  cp_async_commit();
  for (int r = threadIdx.x; r < Ct; r += 256) bes[r] = 1.f - alpha[(size_t)u * g.T + ch.s + r];
  float W[RPG];
  const float* Wb = w.Wst[buf][0] + (size_t)u * F * h;
#pragma unroll
  for (int q = 0; q < RPG; ++q) W[q] = Wb[(size_t)(i0 + q) * h + j];
  cp_async_wait<0>();
  __syncthreads();
  const float* slot0 = w.Ubuf + (size_t)u * g.C * slot_stride + (size_t)i0 * h + j;
  for (int r0 = 0; r0 < Ct; r0 += PD) {
    float cur[PD][RPG];
#pragma unroll
    for (int p = 0; p < PD; ++p) {
      const float* sl = slot0 + (size_t)(r0 + p) * slot_stride;
#pragma unroll
      for (int q = 0; q < RPG; ++q) cur[p][q] = r0 + p < Ct && r0 + p >= rn ? sl[(size_t)q * h] : 0.f;
    }
#pragma unroll
    for (int p = 0; p < PD; ++p) {
      const int r = r0 + p;
      if (r >= Ct) break;
      const float be = bes[r];
      const float* rr = rq + r * (F + 1) + i0;
      float z = 0.f;
#pragma unroll
      for (int q = 0; q < RPG; ++q) {
        if (pre) z += rr[q] * W[q];
        W[q] = be * W[q] + cur[p][q];
        if (!pre) z += rr[q] * W[q];
      }
      part[(r * 8 + grp) * 33 + lane] = z;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < Ct * 32; e += 256) {
    const int r = e >> 5, l = e & 31;
    float z = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) z += part[(r * 8 + k) * 33 + l];
    aq[((size_t)u * g.C + r) * h + jb + l] = siluf_(z);
  }
  float* Wo = w.Wst[buf ^ 1][0] + (size_t)u * F * h;
#pragma unroll
  for (int q = 0; q < RPG; ++q) Wo[(size_t)(i0 + q) * h + j] = W[q];
}

// Pass 2: y_t = r_t + aq_t W2_t.  One warp per row k of W2^T (d x h): lane
// holds columns lane, lane + 32, ... (CPL of them: the warp's shared-memory
// reads of aq_t are conflict-free and its U_t reads coalesced); a shuffle sum
// over the warp gives y_t[k].
template <int CPL>
__global__ void __launch_bounds__(256) k_ns_scan_w2(Geom g, Chunk ch, Work w, int buf, size_t slot_stride,
                                                    const float* alpha, const float* aq, float* y) {
  // W2 decay scan fused with the output read-out.  Warp = output column k,
  // lane = CPL hidden entries; the U_t of PD tokens are loaded together and
  // their PD warp reductions interleave.  The hidden read-outs are staged AW
  // tokens at a time in two buffers (the next window loads during this one),
  // which keeps the CTA at 66 KB of shared memory: more CTAs, and more U_t
  // loads in flight, per SM.
  constexpr int PD = 64 / CPL, AW = 16;   // PD CPL = 64 values in flight per thread
  static_assert(AW % PD == 0, "whole token groups per window");
  extern __shared__ float aqs[];   // [2][AW][h], then [Ct] 1 - alpha
  const int u = blockIdx.y;
  const int lane = threadIdx.x % 32, k = blockIdx.x * 8 + threadIdx.x / 32;
  const int F = g.F, h = g.hidden, d = g.d_v;   // lane holds hidden columns lane + 32 q
  const int Ct = ch.e - ch.s;
  const bool pre = g.readout == ATLAS_READOUT_PRE;   // read out before token r's update
  const int rn = ns_first_row(g, ch);                 // slots before it hold no U_t: U_t = 0
  float* bes = aqs + 2 * AW * h;
  const float* aq_u = aq + (size_t)u * g.C * h;
  // window wd's hidden read-outs by 16-byte cp.async (h % 32 == 0, 16-byte
  // aligned rows), all in flight at once
  auto stage = [&](int wd) {
    const int r0w = wd * AW, nr = Ct - r0w < AW ? Ct - r0w : AW;
    float* dst = aqs + (wd & 1) * AW * h;
    for (int e = 4 * threadIdx.x; e < nr * h; e += 4 * 256) cp_async16(dst + e, aq_u + (size_t)r0w * h + e);
    cp_async_commit();
  };
  stage(0);
  for (int r = threadIdx.x; r < Ct; r += 256) bes[r] = 1.f - alpha[(size_t)u * g.T + ch.s + r];
  float W[CPL];
  const float* Wb = w.Wst[buf][1] + (size_t)u * h * d;   // original orientation [h][d]
#pragma unroll
  for (int q = 0; q < CPL; ++q) W[q] = Wb[(size_t)(lane + 32 * q) * d + k];
  const float* slot0 = w.Ubuf + (size_t)u * g.C * slot_stride + (size_t)F * h + (size_t)k * h + lane;
  for (int wd = 0; wd * AW < Ct; ++wd) {
    if ((wd + 1) * AW < Ct) {
      stage(wd + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* aw = aqs + (wd & 1) * AW * h - (size_t)wd * AW * h;   // indexed by chunk row r
    const int rend = (wd + 1) * AW < Ct ? (wd + 1) * AW : Ct;
    for (int r0 = wd * AW; r0 < rend; r0 += PD) {
      float cur[PD][CPL];
#pragma unroll
      for (int p = 0; p < PD; ++p) {
        const float* sl = slot0 + (size_t)(r0 + p) * slot_stride;
#pragma unroll
        for (int q = 0; q < CPL; ++q) cur[p][q] = r0 + p < rend && r0 + p >= rn ? sl[32 * q] : 0.f;
      }
      float acc[PD];
#pragma unroll
      for (int p = 0; p < PD; ++p) {
        const int r = r0 + p < rend ? r0 + p : rend - 1;
        const float be = bes[r];
        float a = 0.f;
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
          if (r0 + p < rend) {
            if (pre) a += aw[r * h + lane + 32 * q] * W[q];
            W[q] = be * W[q] + cur[p][q];
            if (!pre) a += aw[r * h + lane + 32 * q] * W[q];
          }
        }
        acc[p] = a;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int p = 0; p < PD; ++p) acc[p] += __shfl_xor_sync(0xffffffffu, acc[p], o);
      if (lane == 0)
#pragma unroll
        for (int p = 0; p < PD; ++p) {
          const int r = r0 + p;
          if (r < rend) {
            const size_t yi = ((size_t)u * g.T + ch.s + r) * d + k;
            y[yi] = w.R[((size_t)u * g.T + ch.s + r) * F + k] + acc[p];
          }
        }
    }
    __syncthreads();   // this window's buffer may be restaged
  }
  float* Wo = w.Wst[buf ^ 1][1] + (size_t)u * h * d;
#pragma unroll
  for (int q = 0; q < CPL; ++q) Wo[(size_t)(lane + 32 * q) * d + k] = W[q];
}

bool ns_fused_scan_supported(const Geom& g) {
  if (g.depth != 2 || g.ns_iters <= 0) return false;
  const int F = g.F, h = g.hidden, d = g.d_v;
  if (!(F <= h && h > d)) return false;              // W1 not tall, W2 tall
  if (h % 32 || d % 8 || F % 8) return false;
  if (!((F / 8 == 8) || (F / 8 == 16))) return false;   // row groups of 8 or 16
  if (!((h / 32 == 8) || (h / 32 == 16))) return false; // 8 or 16 columns per lane
  if (g.C > 64) return false;
  return true;
}

cudaError_t ns_fused_scan(const Geom& g, const Chunk& ch, const Work& w, int buf, size_t slot_stride,
                          const float* alpha, float* aq, float* y, cudaStream_t st) {
  const int F = g.F, h = g.hidden, d = g.d_v;
  dim3 g1(h / 32, g.units);
  const size_t sm1 = ((size_t)g.C * (F + 1) + (size_t)g.C * 8 * 33 + g.C) * sizeof(float);
  if (F / 8 == 8) {
    cudaFuncSetAttribute(k_ns_scan_w1<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    k_ns_scan_w1<8><<<g1, 256, sm1, st>>>(g, ch, w, buf, slot_stride, alpha, aq);
  } else {
    cudaFuncSetAttribute(k_ns_scan_w1<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    k_ns_scan_w1<16><<<g1, 256, sm1, st>>>(g, ch, w, buf, slot_stride, alpha, aq);
  }
  const size_t sm2 = ((size_t)2 * 16 * h + (ch.e - ch.s)) * sizeof(float);   // two windows of 16 tokens
  dim3 g2(d / 8, g.units);
  if (h / 32 == 8) {
    cudaFuncSetAttribute(k_ns_scan_w2<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
    k_ns_scan_w2<8><<<g2, 256, sm2, st>>>(g, ch, w, buf, slot_stride, alpha, aq, y);
  } else {
    cudaFuncSetAttribute(k_ns_scan_w2<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
    k_ns_scan_w2<16><<<g2, 256, sm2, st>>>(g, ch, w, buf, slot_stride, alpha, aq, y);
  }
  return cudaGetLastError();
}

}  // namespace atlas

namespace atlas {

// --------------------------------------------- tiled gradient factors
// The window rows' forward, error and backward at the chunk-start weights
// as 64 x 64 register-tiled fp32 GEMMs (tile_gemm), one CTA per (unit,
// 64-wide output block).

// depth 1: dy = 2 gamma (X W - V)
__global__ void __launch_bounds__(256) k_grad1_tiled(Geom g, Chunk ch, Work w, int buf) {
  __shared__ float As[16 * 64], Bs[16 * 64];
  const int u = blockIdx.z, i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  const float* Xw = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
  const float* Vw = w.V + ((size_t)u * g.L + ch.lo + g.n_prev) * g.d_v;
  const float* Gw = w.G + (size_t)u * g.L + ch.lo + g.n_prev;
  const float* W = w.Wst[buf][0] + (size_t)u * g.F * g.d_v;
  float acc[4][4];
  tile_gemm(TileOp{Xw, g.F, 1}, TileOp{W, 1, g.d_v}, ch.nw, g.d_v, g.F, i0, j0, acc, As, Bs);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int a = 0; a < 4; ++a) {
    const int i = i0 + ty * 4 + a;
    if (i >= ch.nw) continue;
    for (int b = 0; b < 4; ++b) {
      const int j = j0 + tx * 4 + b;
      if (j < g.d_v) w.DY[((size_t)u * g.Kw + i) * g.d_v + j] = 2.f * Gw[i] * (acc[a][b] - Vw[(size_t)i * g.d_v + j]);
    }
  }
}

// depth 2, part 1: Z = X W1[:, jb] -> z, a = SiLU(z); partial Yhat = a W2[jb, :]
__global__ void __launch_bounds__(256) k_grad2_fwd(Geom g, Chunk ch, Work w, int buf, float* part) {
  // one CTA per (64 hidden units, 64 window rows, unit): Z and A of its
  // tile, then its hidden block's partial forward output A W2
  __shared__ float As[16 * 64], Bs[16 * 64];
  __shared__ float Ablk[64 * 65];
  const int u = blockIdx.z, i0 = blockIdx.y * 64, jb = blockIdx.x * 64, h = g.hidden;
  const float* Xw = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F;
  const float* W1 = w.Wst[buf][0] + (size_t)u * g.F * h;
  const float* W2 = w.Wst[buf][1] + (size_t)u * h * g.d_v;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int hb = h - jb < 64 ? h - jb : 64;
  {
    float acc[4][4];
    tile_gemm(TileOp{Xw, g.F, 1}, TileOp{W1 + jb, 1, h}, ch.nw, hb, g.F, i0, 0, acc, As, Bs);
    for (int a = 0; a < 4; ++a) {
      const int il = ty * 4 + a, i = i0 + il;
      for (int b = 0; b < 4; ++b) {
        const int j = tx * 4 + b;
        const float z = acc[a][b];
        const float av = siluf_(z);
        if (i < ch.nw && j < hb) {
          const size_t o = ((size_t)u * g.Kw + i) * h + jb + j;
          w.Zpre[o] = z;
          w.Aact[o] = av;
        }
        Ablk[il * 65 + j] = (i < ch.nw && j < hb) ? av : 0.f;
      }
    }
  }
  __syncthreads();
  const int nb = (h + 63) / 64;
  for (int j0 = 0; j0 < g.d_v; j0 += 64) {
    float acc[4][4];
    tile_gemm(TileOp{Ablk, 65, 1}, TileOp{W2 + (size_t)jb * g.d_v, 1, g.d_v}, ch.nw - i0, g.d_v, hb, 0, j0, acc, As,
              Bs);
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + ty * 4 + a;
      if (i >= ch.nw) continue;
      for (int b = 0; b < 4; ++b) {
        const int j = j0 + tx * 4 + b;
        if (j < g.d_v) part[(((size_t)u * nb + blockIdx.x) * g.Kw + i) * g.d_v + j] = acc[a][b];
      }
    }
  }
}

// depth 2, part 2: dy = 2 gamma (X + sum of partials - V)
__global__ void k_grad2_dy(Geom g, Chunk ch, Work w, const float* part) {
  const int u = blockIdx.y;
  const int nb = (g.hidden + 63) / 64;
  const size_t n = (size_t)ch.nw * g.d_v;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e / g.d_v), j = (int)(e % g.d_v);
    const size_t row = (size_t)u * g.L + ch.lo + g.n_prev + i;
    float yh = w.X[row * g.F + j];   // residual (F == d_v)
    for (int b = 0; b < nb; ++b) yh += part[(((size_t)u * nb + b) * g.Kw + i) * g.d_v + j];
    w.DY[((size_t)u * g.Kw + i) * g.d_v + j] = 2.f * w.G[row] * (yh - w.V[row * g.d_v + j]);
  }
}

// depth 2, part 3: dz[:, jb] = (dy W2[jb, :]^T) * SiLU'(z)
__global__ void __launch_bounds__(256) k_grad2_dz(Geom g, Chunk ch, Work w, int buf) {
  __shared__ float As[16 * 64], Bs[16 * 64];
  const int u = blockIdx.z, i0 = blockIdx.y * 64, jb = blockIdx.x * 64, h = g.hidden;
  const float* DYw = w.DY + (size_t)u * g.Kw * g.d_v;
  const float* W2 = w.Wst[buf][1] + (size_t)u * h * g.d_v;
  float acc[4][4];
  tile_gemm(TileOp{DYw, g.d_v, 1}, TileOp{W2 + (size_t)jb * g.d_v, g.d_v, 1}, ch.nw, h - jb < 64 ? h - jb : 64, g.d_v,
            i0, 0, acc, As, Bs);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int a = 0; a < 4; ++a) {
    const int i = i0 + ty * 4 + a;
    if (i >= ch.nw) continue;
    for (int b = 0; b < 4; ++b) {
      const int j = jb + tx * 4 + b;
      if (j < h) {
        const size_t o = ((size_t)u * g.Kw + i) * h + j;
        w.DZ[o] = acc[a][b] * dsiluf_(w.Zpre[o]);
      }
    }
  }
}

size_t grad_part_floats(const Geom& g) {
  return g.depth == 2 ? (size_t)g.units * ((g.hidden + 63) / 64) * g.Kw * g.d_v : 0;
}

cudaError_t grad_tiled(const Geom& g, const Chunk& ch, const Work& w, int buf, cudaStream_t st, int* nl) {
  const int rt = (ch.nw + 63) / 64;
  if (g.depth == 2 && grad_tc_supported(g)) {
    // tensor cores: z, a and per-block partial outputs; dy; dz
    CUDA_CHECK_RET(grad_tc_fwd_launch(g, ch, w, buf, w.gpart, st));
    k_grad2_dy<<<dim3(4, g.units), 256, 0, st>>>(g, ch, w, w.gpart);
    CUDA_CHECK_RET(cudaGetLastError());
    *nl += 2;
    return grad_tc_dz_launch(g, ch, w, buf, st);
  }
  if (g.depth == 1) {
    k_grad1_tiled<<<dim3((g.d_v + 63) / 64, rt, g.units), 256, 0, st>>>(g, ch, w, buf);
    return cudaGetLastError();
  }
  const int nb = (g.hidden + 63) / 64;
  k_grad2_fwd<<<dim3(nb, rt, g.units), 256, 0, st>>>(g, ch, w, buf, w.gpart);
  k_grad2_dy<<<dim3(4, g.units), 256, 0, st>>>(g, ch, w, w.gpart);
  k_grad2_dz<<<dim3(nb, rt, g.units), 256, 0, st>>>(g, ch, w, buf);
  *nl += 2;
  return cudaGetLastError();
}

}  // namespace atlas

namespace atlas {

// ------------------------------------------- projected polynomial features
// out = phi(x) P for 64 token rows per CTA as a register-tiled fp32 GEMM;
// phi is generated tile by tile from the raw rows held in shared memory
// (pair indices of the degree-2 monomials tabulated once per CTA).
__global__ void __launch_bounds__(256) k_features_proj(Geom g, const void* src, const void* cache, int rows_per_unit,
                                                      int from_cache, const void* P, float* out) {
  extern __shared__ float smf[];
  float* xs = smf;                              // [64][d_k + 1]
  float* As = xs + 64 * (g.d_k + 1);            // [16][64] phi tile (k-major)
  float* Bs = As + 16 * 64;                     // [16][64] P tile
  unsigned short* pij = reinterpret_cast<unsigned short*>(Bs + 16 * 64);   // [poly] (i << 8) | j
  const int u = blockIdx.y, r0 = blockIdx.x * 64, d = g.d_k, ld = d + 1;
  for (int e = threadIdx.x; e < 64 * d; e += blockDim.x) {
    const int rr = e / d, k = e % d, row = r0 + rr;
    float val = 0.f;
    if (row < rows_per_unit) {
      if (from_cache && row < g.n_prev) {
        const size_t slot = (size_t)(g.c - 1 - g.n_prev + row);
        val = load_in(cache, ((size_t)u * (g.c - 1) + slot) * d + k, g.qkv_dtype);
      } else {
        const int t = row - (from_cache ? g.n_prev : 0);
        val = load_in(src, ((size_t)u * g.T + t) * d + k, g.qkv_dtype);
      }
    }
    xs[rr * ld + k] = val;
  }
  for (int f = threadIdx.x; f < g.poly; f += blockDim.x) {
    int i = 0, jj = 0;
    if (f > d) {
      int q = f - 1 - d;
      while (q >= d - i) { q -= d - i; ++i; }
      jj = i + q;
    }
    pij[f] = (unsigned short)((i << 8) | jj);
  }
  __syncthreads();
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int f0 = 0; f0 < g.poly; f0 += 16) {
    for (int l = threadIdx.x; l < 16 * 64; l += blockDim.x) {
      const int kk = l / 64, ii = l % 64, f = f0 + kk;
      float ph = 0.f;
      if (f < g.poly) {
        if (f == 0) ph = 1.f;
        else if (f <= d) ph = xs[ii * ld + f - 1];
        else { const unsigned short pr = pij[f]; ph = 0.5f * xs[ii * ld + (pr >> 8)] * xs[ii * ld + (pr & 255)]; }
      }
      As[kk * 64 + ii] = ph;
      Bs[kk * 64 + ii] = (f < g.poly && ii < g.proj_dim) ? load_in(P, (size_t)f * g.proj_dim + ii, g.qkv_dtype) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) av[a] = As[kk * 64 + ty * 4 + a];
#pragma unroll
      for (int b = 0; b < 4; ++b) bv[b] = Bs[kk * 64 + tx * 4 + b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] += av[a] * bv[b];
    }
    __syncthreads();
  }
  for (int a = 0; a < 4; ++a) {
    const int row = r0 + ty * 4 + a;
    if (row >= rows_per_unit) continue;
    for (int b = 0; b < 4; ++b) {
      const int j = tx * 4 + b;
      if (j < g.proj_dim) out[((size_t)u * rows_per_unit + row) * g.F + j] = acc[a][b];
    }
  }
}

size_t features_proj_smem(const Geom& g) {
  return (size_t)(64 * (g.d_k + 1) + 2 * 16 * 64) * sizeof(float) + (size_t)g.poly * sizeof(unsigned short) + 16;
}

bool features_proj_supported(const Geom& g) {
  return g.proj_dim > 0 && g.proj_dim <= 64 && g.p == 2 && g.d_k <= 255 && features_proj_smem(g) <= 200 * 1024;
}

cudaError_t features_proj_launch(const Geom& g, const void* src, const void* cache, int rows, int from_cache,
                                 const void* P, float* out, cudaStream_t st) {
  const size_t sm = features_proj_smem(g);
  cudaFuncSetAttribute(k_features_proj, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  k_features_proj<<<dim3((rows + 63) / 64, g.units), 256, sm, st>>>(g, src, cache, rows, from_cache, P, out);
  return cudaGetLastError();
}

}  // namespace atlas

namespace atlas {

// ------------------------------------------ split dual form, depth 1
// Every product of a depth-1 chunk contracts over the feature axis F (561
// for degree-2 features of 32-dim keys) except the small window term, so
// the chunk is cut along F.  For each (64-feature slice, unit):
//   PW = R W, PS = R S, PX = R X^T, PG = X W    (restricted to the slice)
// A combine kernel sums the slices, runs the chunk's coefficient scans and
// forms dy_i = 2 gamma_i (x_i W - v_i), M = Cw (.) R X^T and
//   y_t = B_t (R W)_t + D_t (R S)_t - (M dY)_t.
// A step kernel, again one CTA per (slice, unit), updates the slice's rows
// of the state,
//   S' = A_e S - X^T diag(cs_e) dY,  W' = B_e W + D_e S - X^T diag(cw_e) dY,
// and, keeping them in shared memory, forms the next chunk's partial
// products.  Two launches per chunk.

// floats per (unit, slice) of partial products
__host__ __device__ inline size_t dual1_part_floats(const Geom& g) {
  return 2 * (size_t)g.C * g.d_v + (size_t)g.C * g.Kw + (size_t)g.Kw * g.d_v;
}

// acc[a][b] = sum_{k < K} A(ty*4+a, k) B(k, tx*4+b) over shared-memory
// operands stored k-major: A(i, k) = At[k * lda + i], B(k, j) = B[k * ldb + j]
// (lda, ldb and both bases multiples of 4 floats: one 16-byte load per
// operand and k)
__device__ __forceinline__ void smem_gemm(const float* At, int lda, const float* B, int ldb, int K,
                                          float acc[4][4], int tid) {
  const int tx = tid % 16, ty = tid / 16;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
  for (int k = 0; k < K; ++k) {
    const float4 av = *reinterpret_cast<const float4*>(At + k * lda + ty * 4);
    const float4 bv = *reinterpret_cast<const float4*>(B + k * ldb + tx * 4);
    const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] += ar[a] * br[b];
  }
}

// store rows [r0, r0 + 64) x cols [0, 64) of acc into out (row stride ld),
// rows < nr and cols < nc only
__device__ __forceinline__ void store_tile(float* out, int ld, int r0, int nr, int nc, const float acc[4][4],
                                           int tid) {
  const int tx = tid % 16, ty = tid / 16;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int r = r0 + ty * 4 + a;
    if (r >= nr) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int c = tx * 4 + b;
      if (c < nc) out[(size_t)r * ld + c] = acc[a][b];
    }
  }
}


// shared-memory slices, all k-major for smem_gemm: R transposed [f][t]
// (row stride 68), X transposed [f][i] (row stride 132), X [i][f] (row
// stride 68), W and S [f][j] (row stride 64)
constexpr int kRtF = 64 * 68, kXtF = 64 * 132, kXrF = 128 * 68, kWsF = 64 * 64;
constexpr size_t kDual1PartSmem = (size_t)(kRtF + kXtF + 2 * kWsF) * sizeof(float);
constexpr size_t kDual1StepSmem = kDual1PartSmem + (size_t)(kXrF + 2 * 128 * 64) * sizeof(float);

// issue copies of the R rows of chunk ch and its window rows of X,
// features [f0, f0 + 64), both transposed
__device__ void dual1_load_rx(const Geom& g, const Chunk& ch, const Work& w, int u, int f0, float* Rt, float* Xt) {
  const int Ct = ch.e - ch.s, nf = min(64, g.F - f0);
  const float* Rw = w.R + ((size_t)u * g.T + ch.s) * g.F + f0;
  const float* Xw = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F + f0;
  for (int l = threadIdx.x; l < 64 * 64; l += blockDim.x) {
    const int r = l / 64, c = l % 64;
    cp_async4(&Rt[c * 68 + r], Rw + (size_t)r * g.F + c, r < Ct && c < nf, w.R);
  }
  for (int l = threadIdx.x; l < 128 * 64; l += blockDim.x) {
    const int i = l / 64, f = l % 64;
    cp_async4(&Xt[f * 132 + i], Xw + (size_t)i * g.F + f, i < ch.nw && f < nf, w.X);
  }
}

// issue copies of rows [f0, f0 + 64) of the state matrices
__device__ void dual1_load_ws(const Geom& g, const Work& w, int buf, int u, int f0, float* Ws, float* Ss) {
  const int nf = min(64, g.F - f0), dv = g.d_v;
  const size_t so = ((size_t)u * g.F + f0) * dv;
  for (int l = threadIdx.x; l < 64 * 64; l += blockDim.x) {
    const int r = l / 64, c = l % 64;
    const bool ok = r < nf && c < dv;
    cp_async4(&Ws[l], w.Wst[buf][0] + so + (size_t)r * dv + c, ok, w.Wst[buf][0]);
    cp_async4(&Ss[l], w.Sst[buf][0] + so + (size_t)r * dv + c, ok, w.Sst[buf][0]);
  }
}

__device__ void dual1_partials_smem(const Geom& g, const Chunk& ch, const float* Rt, const float* Xt,
                                    const float* Ws, const float* Ss, float* pb) {
  const int Ct = ch.e - ch.s, nw = ch.nw, dv = g.d_v;
  float* PW = pb;
  float* PS = PW + (size_t)g.C * dv;
  float* PX = PS + (size_t)g.C * dv;
  float* PG = PX + (size_t)g.C * g.Kw;
  float acc[4][4];
  smem_gemm(Rt, 68, Ws, 64, 64, acc, threadIdx.x);
  store_tile(PW, dv, 0, Ct, dv, acc, threadIdx.x);
  smem_gemm(Rt, 68, Ss, 64, 64, acc, threadIdx.x);
  store_tile(PS, dv, 0, Ct, dv, acc, threadIdx.x);
  for (int i0 = 0; i0 < nw; i0 += 64) {
    smem_gemm(Rt, 68, Xt + i0, 132, 64, acc, threadIdx.x);
    store_tile(PX + i0, g.Kw, 0, Ct, nw - i0, acc, threadIdx.x);
    smem_gemm(Xt + i0, 132, Ws, 64, 64, acc, threadIdx.x);
    store_tile(PG, dv, i0, nw, dv, acc, threadIdx.x);
  }
}

// partial products of the first chunk, from the state in global memory
__global__ void __launch_bounds__(256) k_dual1_partials(Geom g, Chunk ch, Work w, int buf, float* part) {
  extern __shared__ __align__(16) float sm[];
  float* Rt = sm;
  float* Xt = Rt + kRtF;
  float* Ws = Xt + kXtF;
  float* Ss = Ws + kWsF;
  const int kb = blockIdx.x, u = blockIdx.y, f0 = kb * 64;
  dual1_load_ws(g, w, buf, u, f0, Ws, Ss);
  dual1_load_rx(g, ch, w, u, f0, Rt, Xt);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  dual1_partials_smem(g, ch, Rt, Xt, Ws, Ss, part + ((size_t)u * gridDim.x + kb) * dual1_part_floats(g));
}

// The gate scans depend on theta, eta, alpha only, so every chunk's are
// formed up front, one CTA per (chunk, unit):
//   Cs_t[i] = eta_t Cs_{t-1}[i] + theta_t [t in window of row i],
//   Cw_t[i] = (1 - alpha_t) Cw_{t-1}[i] + Cs_t[i],
//   A_t = prod eta, B_t = prod (1 - alpha), D_t = (1 - alpha_t) D_{t-1} + A_t.
__global__ void __launch_bounds__(160) k_dual1_coef_all(Geom g, const float* theta, const float* eta,
                                                         const float* alpha, float* coef, CoefLayout L) {
  __shared__ float th[64], et[64], be[64];
  const int n = blockIdx.x, u = blockIdx.y;
  // pre-update read-out: token r reads the state after token r - 1 (the
  // chunk-start state for r = 0: Cw = 0, B = 1, D = 0)
  const bool pre = g.readout == ATLAS_READOUT_PRE;
  const Chunk ch = dual1_chunk_at(g, n * g.C);
  const int Ct = g.C;
  for (int r = threadIdx.x; r < Ct; r += blockDim.x) {
    th[r] = theta[(size_t)u * g.T + ch.s + r];
    et[r] = eta[(size_t)u * g.T + ch.s + r];
    be[r] = 1.f - alpha[(size_t)u * g.T + ch.s + r];
  }
  __syncthreads();
  float* cb = coef + ((size_t)u * gridDim.x + n) * L.floats(g.C);
  float* Cw = cb;
  float* cse = cb + L.o_cs(g.C);
  float* cwe = cb + L.o_cw(g.C);
  float* Bt = cb + L.o_bt(g.C);
  float* Dt = cb + L.o_dt(g.C);
  float* ABD = cb + L.o_abd(g.C);
  if (threadIdx.x < ch.nw) {
    const int i = threadIdx.x, ti = ch.lo + i;
    float cs = 0.f, cw = 0.f;
    for (int r = 0; r < Ct; ++r) {
      const int t = ch.s + r;
      const bool in_win = ti <= t && t <= ti + g.c - 1;
      const float cw_prev = cw;
      cs = et[r] * cs + (in_win ? th[r] : 0.f);
      cw = be[r] * cw + cs;
      Cw[(size_t)r * L.kws + i] = pre ? cw_prev : cw;   // read-out weights of token r
    }
    cse[i] = cs;
    cwe[i] = cw;
  } else if (threadIdx.x < L.kws) {   // padding columns past the window
    const int i = threadIdx.x;
    for (int r = 0; r < Ct; ++r) Cw[(size_t)r * L.kws + i] = 0.f;
    cse[i] = 0.f;
    cwe[i] = 0.f;
  } else if (threadIdx.x == blockDim.x - 1) {
    float Ap = 1.f, Bp = 1.f, Dp = 0.f;
    for (int r = 0; r < Ct; ++r) {
      const float Bprev = Bp, Dprev = Dp;
      Ap *= et[r];
      Bp *= be[r];
      Dp = be[r] * Dp + Ap;
      Bt[r] = pre ? Bprev : Bp;
      Dt[r] = pre ? Dprev : Dp;
    }
    for (int r = Ct; r < L.cp; ++r) {
      Bt[r] = 0.f;
      Dt[r] = 0.f;
    }
    ABD[0] = Ap;
    ABD[1] = Bp;
    ABD[2] = Dp;
    ABD[3] = 0.f;
  }
}

// Sum of the slices' partial products, one thread per element of a unit's
// block, with the elementwise steps that need only that element:
//   PW, PS copied;  M[t][i] = Cw_t[i] (R X^T)[t][i];
//   dy[i][j] = 2 gamma_i ((X W)[i][j] - v_i[j]) and its cs_e / cw_e scalings.
__global__ void __launch_bounds__(256) k_dual1_reduce(Geom g, Chunk ch, int n, Work w, const float* part,
                                                       const float* coef, float* red, float* dys) {
  const int u = blockIdx.y;
  const size_t per = dual1_part_floats(g);
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= per) return;
  const int ks = (g.F + 63) / 64, dv = g.d_v, Kw = g.Kw;
  const size_t oX = 2 * (size_t)g.C * dv, oG = oX + (size_t)g.C * Kw;
  // rows past the chunk's window were never written: skip them
  if (e >= oX && e < oG && (int)((e - oX) % Kw) >= ch.nw) return;
  if (e >= oG && (int)((e - oG) / dv) >= ch.nw) return;
  const float* p = part + (size_t)u * ks * per + e;
  float s = 0.f;
#pragma unroll 16
  for (int kb = 0; kb < ks; ++kb) s += p[kb * per];
  float* ru = red + (size_t)u * per;
  if (e < oX) {
    ru[e] = s;
  } else if (e < oG) {
    const float* Cw = coef + ((size_t)u * (g.T / g.C) + n) * dual1_coef_floats(g);
    ru[e] = Cw[e - oX] * s;
  } else {
    const float* cb = coef + ((size_t)u * (g.T / g.C) + n) * dual1_coef_floats(g);
    const float* cse = cb + (size_t)g.C * Kw;
    const float* cwe = cse + Kw;
    const int i = (int)((e - oG) / dv), j = (int)((e - oG) % dv);
    const size_t row = (size_t)u * g.L + ch.lo + g.n_prev + i;
    const float d = 2.f * w.G[row] * (s - w.V[row * dv + j]);
    ru[e] = d;
    dys[((size_t)u * 2 + 0) * Kw * dv + (size_t)i * dv + j] = cse[i] * d;
    dys[((size_t)u * 2 + 1) * Kw * dv + (size_t)i * dv + j] = cwe[i] * d;
  }
}

// y_t = B_t (R W)_t + D_t (R S)_t - (M dY)_t; one CTA per (16 columns,
// 16 tokens, unit)
__global__ void __launch_bounds__(256) k_dual1_readout(Geom g, Chunk ch, int n, const float* red,
                                                        const float* coef, float* y) {
  __shared__ float M[16][129];
  __shared__ float Dy[128][17];
  const int jb = blockIdx.x * 16, tb = blockIdx.y * 16, u = blockIdx.z;
  const int Ct = ch.e - ch.s, nw = ch.nw, dv = g.d_v, Kw = g.Kw;
  const size_t per = dual1_part_floats(g);
  const float* ru = red + (size_t)u * per;
  const size_t oS = (size_t)g.C * dv, oX = 2 * oS, oG = oX + (size_t)g.C * Kw;
  for (int l = threadIdx.x; l < nw * 16; l += blockDim.x) {
    const int i = l >> 4, jj = l & 15;
    Dy[i][jj] = jb + jj < dv ? ru[oG + (size_t)i * dv + jb + jj] : 0.f;
  }
  {
    const int i = threadIdx.x & 127;
    if (i < nw)
      for (int tt = threadIdx.x >> 7; tt < 16; tt += 2)
        M[tt][i] = tb + tt < Ct ? ru[oX + (size_t)(tb + tt) * Kw + i] : 0.f;
  }
  __syncthreads();
  const int tt = threadIdx.x / 16, jj = threadIdx.x % 16, t = tb + tt, j = jb + jj;
  if (t >= Ct || j >= dv) return;
  const float* cb = coef + ((size_t)u * (g.T / g.C) + n) * dual1_coef_floats(g);
  const float* Bt = cb + (size_t)g.C * Kw + 2 * (size_t)Kw;
  const float* Dt = Bt + g.C;
  float c = 0.f;
  for (int i = 0; i < nw; ++i) c += M[tt][i] * Dy[i][jj];
  y[((size_t)u * g.T + ch.s + t) * dv + j] =
      Bt[t] * ru[(size_t)t * dv + j] + Dt[t] * ru[oS + (size_t)t * dv + j] - c;
}

// chunk-end state of one 64-feature slice, then (if there is a next chunk)
// that slice's partial products of the next chunk from the new state.
// 512 threads: the two 256-thread halves take different products.
__global__ void __launch_bounds__(512) k_dual1_step(Geom g, Chunk ch, Chunk nx, int has_next, int n, Work w,
                                                     int buf, const float* coef, const float* dys, float* part) {
  extern __shared__ __align__(16) float sm[];
  float* Rt = sm;          // next chunk's R, transposed
  float* Xt = Rt + kRtF;   // next chunk's X, transposed
  float* Ws = Xt + kXtF;
  float* Ss = Ws + kWsF;
  float* Xr = Ss + kWsF;   // this chunk's X [i][f]
  float* Dc = Xr + kXrF;   // [2][128][64]: cs_e dy, cw_e dy
  const int kb = blockIdx.x, u = blockIdx.y, f0 = kb * 64, dv = g.d_v, nw = ch.nw;
  const int nf = min(64, g.F - f0);
  const int half = threadIdx.x >> 8, tid = threadIdx.x & 255;
  const size_t so = ((size_t)u * g.F + f0) * dv;
  dual1_load_ws(g, w, buf, u, f0, Ws, Ss);
  const float* Xw = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F + f0;
  for (int l = threadIdx.x; l < 128 * 64; l += blockDim.x) {
    const int i = l / 64, f = l % 64;
    cp_async4(&Xr[i * 68 + f], Xw + (size_t)i * g.F + f, i < nw && f < nf, w.X);
    for (int h = 0; h < 2; ++h)
      cp_async4(&Dc[h * 128 * 64 + l], dys + (((size_t)u * 2 + h) * g.Kw + i) * dv + f, i < nw && f < dv, dys);
  }
  cp_async_commit();
  if (has_next) dual1_load_rx(g, nx, w, u, f0, Rt, Xt);
  cp_async_commit();
  const float* ABD = coef + ((size_t)u * (g.T / g.C) + n) * dual1_coef_floats(g) + (size_t)g.C * g.Kw +
                     2 * (size_t)g.Kw + 2 * (size_t)g.C;
  const float Ae = ABD[0], Be = ABD[1], De = ABD[2];
  cp_async_wait<1>();
  __syncthreads();
  float acc[4][4];
  // half 0: X^T (cs_e dy) -> S;  half 1: X^T (cw_e dy) -> W
  smem_gemm(Xr, 68, Dc + half * 128 * 64, 64, nw, acc, tid);
  const int tx = tid % 16, ty = tid / 16;
  float sn[4][4];
  if (half == 0) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) sn[a][b] = Ae * Ss[(ty * 4 + a) * 64 + tx * 4 + b] - acc[a][b];
  } else {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int o = (ty * 4 + a) * 64 + tx * 4 + b;
        sn[a][b] = Be * Ws[o] + De * Ss[o] - acc[a][b];
      }
  }
  __syncthreads();   // every read of the old S is done
  float* dst = half == 0 ? w.Sst[buf ^ 1][0] : w.Wst[buf ^ 1][0];
  float* sdst = half == 0 ? Ss : Ws;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int f = ty * 4 + a;
    if (f >= nf) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int j = tx * 4 + b;
      if (j >= dv) continue;
      dst[so + (size_t)f * dv + j] = sn[a][b];
      sdst[f * 64 + j] = sn[a][b];
    }
  }
  cp_async_wait<0>();
  if (!has_next) return;
  __syncthreads();
  const int Ct = nx.e - nx.s, nwn = nx.nw;
  float* pb = part + ((size_t)u * gridDim.x + kb) * dual1_part_floats(g);
  float* PW = pb;
  float* PS = PW + (size_t)g.C * dv;
  float* PX = PS + (size_t)g.C * dv;
  float* PG = PX + (size_t)g.C * g.Kw;
  if (half == 0) {
    smem_gemm(Rt, 68, Ws, 64, 64, acc, tid);
    store_tile(PW, dv, 0, Ct, dv, acc, tid);
    for (int i0 = 0; i0 < nwn; i0 += 64) {
      smem_gemm(Rt, 68, Xt + i0, 132, 64, acc, tid);
      store_tile(PX + i0, g.Kw, 0, Ct, nwn - i0, acc, tid);
    }
  } else {
    smem_gemm(Rt, 68, Ss, 64, 64, acc, tid);
    store_tile(PS, dv, 0, Ct, dv, acc, tid);
    for (int i0 = 0; i0 < nwn; i0 += 64) {
      smem_gemm(Xt + i0, 132, Ws, 64, 64, acc, tid);
      store_tile(PG, dv, i0, nwn, dv, acc, tid);
    }
  }
}

cudaError_t dual1_coef_launch(const Geom& g, const GenericIO& io, float* coef, CoefLayout L, cudaStream_t st) {
  k_dual1_coef_all<<<dim3(g.T / g.C, g.units), 160, 0, st>>>(g, io.theta, io.eta, io.alpha, coef, L);
  return cudaGetLastError();
}

cudaError_t values_launch(const Geom& g, const Work& w, const GenericIO& io, cudaStream_t st) {
  k_values<<<dim3(g.L, g.units), 128, 0, st>>>(g, io.v, io.win_v, io.gamma, io.win_gamma, w.V, w.G);
  return cudaGetLastError();
}

bool dual1_split_supported(const Geom& g) {
  return g.depth == 1 && g.ns_iters == 0 && g.update == ATLAS_UPDATE_PER_TOKEN && g.Kw <= 128 && g.C <= 64 &&
         g.d_v <= 64;
}

size_t dual1_split_floats(const Geom& g, size_t units, int T) {
  return units * (2 * (size_t)g.Kw * g.d_v + (size_t)((g.F + 63) / 64 + 1) * dual1_part_floats(g) +
                  (size_t)(T / g.C) * coef_layout_tc(g).floats(g.C));   // covers both layouts
}

cudaError_t dual1_split(const Geom& g, const Chunk& ch, const Work& w, const GenericIO& io, int buf,
                        cudaStream_t st, int* nl) {
  const int ks = (g.F + 63) / 64, Ct = ch.e - ch.s, n = ch.s / g.C;
  const size_t per = dual1_part_floats(g);
  float* dys = w.gpart;
  float* part = dys + (size_t)g.units * 2 * g.Kw * g.d_v;
  float* red = part + (size_t)g.units * ks * per;
  float* coef = red + (size_t)g.units * per;
  if (ch.s == 0) {
    k_dual1_coef_all<<<dim3(g.T / g.C, g.units), 160, 0, st>>>(g, io.theta, io.eta, io.alpha, coef,
                                                              coef_layout_simt(g));
    cudaFuncSetAttribute(k_dual1_partials, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDual1PartSmem);
    k_dual1_partials<<<dim3(ks, g.units), 256, kDual1PartSmem, st>>>(g, ch, w, buf, part);
    *nl += 2;
  }
  k_dual1_reduce<<<dim3((unsigned)((per + 255) / 256), g.units), 256, 0, st>>>(g, ch, n, w, part, coef, red, dys);
  k_dual1_readout<<<dim3((g.d_v + 15) / 16, (Ct + 15) / 16, g.units), 256, 0, st>>>(g, ch, n, red, coef, io.y);
  const int has_next = ch.e < g.T;
  const Chunk nx = dual1_chunk_at(g, has_next ? ch.e : ch.s);
  cudaFuncSetAttribute(k_dual1_step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDual1StepSmem);
  k_dual1_step<<<dim3(ks, g.units), 512, kDual1StepSmem, st>>>(g, ch, nx, has_next, n, w, buf, coef, dys, part);
  *nl += 3;
  return cudaGetLastError();
}

}  // namespace atlas
