// Shared device/host definitions of the memory-layer kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/atlas_mem.h"

namespace atlas {

// Muon quintic Newton-Schulz coefficients and the Frobenius-normalisation eps
// (atlas-torch README, "Atlas Extensions": Muon / Newton-Schulz).
constexpr float kNsA = 3.4445f;
constexpr float kNsB = -4.7750f;
constexpr float kNsC = 2.0315f;
constexpr float kNsEps = 1e-7f;

// Problem geometry shared by every kernel of one forward call.
struct Geom {
  int depth, d_k, d_v, hidden, C, c, p, proj_dim, ns_iters, qkv_dtype;
  int F;          // memory input width (d_k, poly width, or proj_dim)
  int poly;       // width of the monomial expansion (d_k when p == 1)
  int units;      // B * H
  int T;          // tokens of this call
  int n_prev;     // cached tokens in front of this call (win_len)
  int L;          // key rows per unit = n_prev + T
  int Kw;         // max window rows of one chunk = C + c - 1
  int rows[2], cols[2], nmat;
  int readout;    // ATLAS_READOUT_POST / ATLAS_READOUT_PRE
  int ns_target;  // ATLAS_NS_MOMENTUM / ATLAS_NS_SURPRISE
  int update;     // ATLAS_UPDATE_PER_TOKEN / ATLAS_UPDATE_CHUNKWISE
};

// Per-chunk indices: the chunk covers tokens [s, e) of the call; its Omega
// windows reach back to token lo (>= -n_prev), i.e. key rows lo + n_prev ...
struct Chunk {
  int s, e, lo, nw;  // nw = e - lo window rows
};

// Chunk of the call starting at token s (s a multiple of C).
__host__ __device__ inline Chunk dual1_chunk_at(const Geom& g, int s) {
  Chunk c;
  c.s = s;
  c.e = s + g.C;
  c.lo = s - g.c + 1;
  if (c.lo < -g.n_prev) c.lo = -g.n_prev;
  c.nw = c.e - c.lo;
  return c;
}

// Layout of one (unit, chunk) coefficient block of the depth-1 paths:
// Cw [C][kws], cs_e [kws], cw_e [kws], B_t [cp], D_t [cp], (A_e, B_e, D_e,
// pad), row stride kws >= Kw, cp >= C; entries past the chunk's window rows
// or tokens are zero.  Cw, B_t, D_t are the read-out's (shifted by one token
// in pre-update mode); cs_e, cw_e, A_e, B_e, D_e the chunk-end state's.
struct CoefLayout {
  int kws, cp;
  __host__ __device__ size_t floats(int C) const { return (size_t)C * kws + 2 * (size_t)kws + 2 * (size_t)cp + 4; }
  __host__ __device__ size_t o_cs(int C) const { return (size_t)C * kws; }
  __host__ __device__ size_t o_cw(int C) const { return o_cs(C) + kws; }
  __host__ __device__ size_t o_bt(int C) const { return o_cw(C) + kws; }
  __host__ __device__ size_t o_dt(int C) const { return o_bt(C) + cp; }
  __host__ __device__ size_t o_abd(int C) const { return o_dt(C) + cp; }
};
// the fp32 split path's: unpadded
__host__ __device__ inline CoefLayout coef_layout_simt(const Geom& g) { return CoefLayout{g.Kw, g.C}; }
// the tensor-core path's: rows of 16-byte multiples (16-byte copies)
__host__ __device__ inline CoefLayout coef_layout_tc(const Geom& g) {
  return CoefLayout{(g.Kw + 15) / 16 * 16, (g.C + 3) / 4 * 4};
}
__host__ __device__ inline size_t dual1_coef_floats(const Geom& g) { return coef_layout_simt(g).floats(g.C); }

// First token of a chunk (0-based in the chunk) whose momentum goes through
// Newton-Schulz: every token under the per-token rule; under the chunk-wise
// rule the memory changes once per chunk, so only the last token's.  The
// tokens before it add U = 0 to the decay scans.
__host__ __device__ __forceinline__ int ns_first_row(const Geom& g, const Chunk& ch) {
  return g.update == ATLAS_UPDATE_CHUNKWISE ? ch.e - ch.s - 1 : 0;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ float load_in(const void* p, size_t i, int dtype) {
  return dtype == ATLAS_BF16 ? bf16_to_f32(((const uint16_t*)p)[i]) : ((const float*)p)[i];
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + __expf(-z)); }
__device__ __forceinline__ float siluf_(float z) { return z * sigmoidf_(z); }
__device__ __forceinline__ float dsiluf_(float z) {
  float s = sigmoidf_(z);
  return s * (1.f + z * (1.f - s));
}

// Workspace pointers of one forward call (all fp32, device).
struct Work {
  float* X;       // [units][L][F]     key features (cache rows first)
  float* V;       // [units][L][d_v]   values
  float* G;       // [units][L]        Omega weights
  float* R;       // [units][T][F]     query features
  float* Wst[2][2];  // [buffer][matrix] state W, ping-pong by chunk parity
  float* Sst[2][2];  // [buffer][matrix] state S
  // per-chunk factors of the window rows (Kw rows max)
  float* Zpre;    // depth 2: [units][Kw][hidden] pre-activation z_i
  float* Aact;    // depth 2: [units][Kw][hidden] a_i = SiLU(z_i)
  float* DZ;      // depth 2: [units][Kw][hidden] dz_i (gamma folded in)
  float* DY;      // [units][Kw][d_v] dy_i = 2 gamma_i (yhat_i - v_i)
  float* Cs;      // [units][C][Kw]  momentum coefficient of row i in S_t
  float* Cw;      // [units][C][Kw]  coefficient of row i in W_t
  float* Ap;      // [units][C]  prod eta (s..t)
  float* Bp;      // [units][C]  prod (1 - alpha) (s..t)
  float* Dp;      // [units][C]  coefficient of S_bar in W_t
  float* Ubuf;    // NS path: [units][C][sum_m rows*cols] U_t then W_t (X orientation)
  float* gpart;   // depth 2: per hidden block partial forward outputs [units][h/64][Kw][d_v];
                  // depth 1: cs_e dy and cw_e dy [units][2][Kw][d_v], then per
                  // (unit, 64-feature slice) partial products R W, R S, R X^T, X W,
                  // then per (unit, chunk) gate-scan coefficients
  float* surp;    // Newton-Schulz on the surprise: Gram matrices, c x c cores,
                  // banded coefficient matrices (k_surprise.cu)
  float* aeff;    // chunk-wise update with Newton-Schulz: [units][T] the decay
                  // each token applies (0, the chunk's mean alpha at its last token)
  void* Pt;       // tensor-core projected features: P transposed, bf16 [proj][monomials
                  // padded to 64] (k_features_tc.cu)
  int* status;    // device status word
};

// Pointers of one call that the generic kernels read (device).
struct GenericIO {
  const void *q, *k, *v, *P, *win_k, *win_v;
  const float *theta, *eta, *alpha, *gamma, *win_gamma;
  float* y;
};

// generic fp32 path (k_generic.cu)
cudaError_t generic_prepare(const Geom& g, const Work& w, const GenericIO& io, cudaStream_t st, int* nl);
cudaError_t generic_chunk(const Geom& g, const Chunk& ch, const Work& w, const GenericIO& io, int buf,
                          cudaStream_t st, int* nl);
cudaError_t generic_cache_out(const Geom& g, const GenericIO& io, float* tmp, void* k_out, void* v_out,
                              float* g_out, cudaStream_t st, int* nl);
size_t generic_smem_readout(const Geom& g);
size_t generic_smem_ns(const Geom& g, int m);
size_t grad_part_floats(const Geom& g);
size_t dual1_split_floats(const Geom& g, size_t units, int T);
// every chunk's gate-scan coefficient block of the depth-1 paths, up front
cudaError_t dual1_coef_launch(const Geom& g, const GenericIO& io, float* coef, CoefLayout L, cudaStream_t st);
// values and Omega weights of every key row into the workspace (V, G)
cudaError_t values_launch(const Geom& g, const Work& w, const GenericIO& io, cudaStream_t st);

// depth-1 memory on polynomial features on the tensor cores, one persistent
// launch per call (k_dual1_tc.cu)
bool dual1_tc_supported(const Geom& g);
bool dual1_tc_inputs_ok(const GenericIO& io);
cudaError_t dual1_tc_launch(const Geom& g, const Work& w, const GenericIO& io, const float* coef, int fbuf,
                            cudaStream_t st);

// Newton-Schulz on the windowed surprise (k_surprise.cu)
size_t surprise_floats(const Geom& g, size_t units);
// offsets (floats) inside one unit's surprise scratch: the read-out's band of
// Mw per token [nmat][C][Kw][2c-1] and Ms_e R, Mw_e R [nmat][2][Kw][maxcols]
struct SurpOff {
  size_t per_unit, mwb, rp, g2;   // floats: per unit, then offsets inside a unit's part
  int maxcols;
};
SurpOff surprise_offsets(const Geom& g);
// the read-out and the chunk-end state of the surprise path on the tensor
// cores (k_surprise_tc.cu)
bool surprise_tc_supported(const Geom& g);
cudaError_t surprise_tc_readout(const Geom& g, const Chunk& ch, const Work& w, int buf, float* y, cudaStream_t st);
cudaError_t surprise_tc_state(const Geom& g, const Chunk& ch, const Work& w, int buf, cudaStream_t st);
cudaError_t surprise_chunk(const Geom& g, const Chunk& ch, const Work& w, const float* theta, const float* eta,
                           const float* alpha, float* y, int buf, cudaStream_t st, int* nl);
int num_sms();

// gradient factors of the depth-2 memory on the tensor cores (k_grad_tc.cu)
bool grad_tc_supported(const Geom& g);
cudaError_t grad_tc_fwd_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, float* part, cudaStream_t st);
cudaError_t grad_tc_dz_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, cudaStream_t st);

// projected polynomial features on the tensor cores (k_features_tc.cu)
bool features_tc_supported(const Geom& g);
size_t features_tc_scratch_bytes(const Geom& g);
cudaError_t features_tc_prepare(const Geom& g, const void* P, void* Pt, cudaStream_t st);
cudaError_t features_tc_launch(const Geom& g, const void* src, const void* cache, int rows, int from_cache,
                               const void* Pt, float* out, int* status, cudaStream_t st);

// fused tensor-core MLP memory without Newton-Schulz (k_mlp_tc.cu)
bool mlp_tc_supported(const Geom& g);
cudaError_t mlp_tc_launch(const Geom& g, const void* q, const void* k, const void* v, const float* theta,
                          const float* eta, const float* alpha, const float* gamma, const float* const* W0,
                          const float* const* S0, float* y, float* const* W_out, float* const* S_out, int* status,
                          cudaStream_t st, int Tst = 0);   // Tst: token stride between units (0: g.T)

// tensor-core Newton-Schulz (k_ns_tc.cu)
bool ns_tc_supported(const Geom& g);
cudaError_t ns_tc_state_in(const Geom& g, int m, const float* src, float* dst, cudaStream_t st);
cudaError_t ns_tc_state_out(const Geom& g, int m, const float* src, float* dst, cudaStream_t st);
cudaError_t ns_tc_launch(const Geom& g, const Chunk& ch, const Work& w, int buf, size_t slot_stride, int num_sms,
                         const float* theta, const float* eta, cudaStream_t st);

}  // namespace atlas
