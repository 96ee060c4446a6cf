// Matrix memory on polynomial features (depth 1) on the tensor cores, one
// persistent launch per call with the state on chip.
//
// The memory is M(x) = phi(x) W with W of F x d_v, phi the degree-p monomial
// map [1, x_i, x_i x_j / 2] of the keys (atlas-torch README, "Atlas
// Extensions": Polynomial Features; ATLAS summary, Sec. 3.1), trained by the
// Omega rule over a window of c keys with momentum and decay (ATLAS summary,
// Sec. 3.2, Omega rule; titans-pytorch-mlx README, "Core Equations", Eq.
// 10-14).  In the chunked form every window gradient is taken at the
// chunk-start state W^, S^:
//   dy_i = 2 gamma_i (X_i W^ - v_i)                       (window rows i)
//   S_t  = A_t S^ - sum_i Cs_t[i] X_i^T dy_i
//   W_t  = B_t W^ + D_t S^ - sum_i Cw_t[i] X_i^T dy_i
//   y_t  = R_t W_t = B_t (R W^)_t + D_t (R S^)_t - sum_i Cw_t[i] (R_t . X_i) dy_i
// with R the chunk's query features and the gate products A, B, D, Cs, Cw
// formed up front (k_dual1_coef_all).
//
// Layout: one cluster of NC CTAs (NC <= 8, the fewest with NC * 96 >= F) per
// (batch, head) unit; CTA q owns features [q FS, q FS + FS) of W and S for
// the whole call: fp32 masters in TMEM, transposed (row j of W^T in the
// M = 64 accumulator lanes), and split-bf16 copies (hi + lo) in shared
// memory as MMA operands.  The monomials are generated in shared memory
// from the raw bf16 keys and queries; a product of two bf16 values (times
// 1/2) has at most 16 significant bits, so its hi + lo split is exact.
//
// Per chunk, on each CTA:
//  1. generate the slice's R (C x FS) and window X (Kw x FS) tiles;
//  2. tensor cores: [R W^ | R S^ | R X^T] (M = 64, N = 128 + Kw) and X W^
//     (M = 128, N = 64), each as hi hi' + hi lo' + lo hi' (fp32 in TMEM);
//  3. the slice's partials go to their owners in the cluster (distributed
//     shared memory): rows t of B_t RW + D_t RS and of R X^T, rows i of X W^;
//  4. owners sum the NC slices in rank order, form dy rows (broadcast to
//     every CTA) and M = Cw * (R X^T) rows;
//  5. tensor cores: (cs_e dY)^T X, then (cw_e dY)^T X, for the chunk-end
//     state, while the owners form y_t = Yp_t - (M dY)_t for their rows;
//  6. S' = A_e S^ - .., W' = B_e W^ + D_e S^ - .. into the TMEM masters and
//     the operand copies.
// Two cluster barriers per chunk order the exchanges.  Every mbarrier wait
// is bounded; a wait that gives up sets the status word and the CTA keeps
// the loop's barrier schedule without issuing further MMAs.
#include <cuda_bf16.h>

#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {
namespace {

constexpr int NT = 256;                 // 8 warps: two per TMEM sub-partition
constexpr int FSM = 96, KWM = 80;       // max features per CTA, max window rows (padded)
constexpr int RAWB = 80;                // bytes per raw input row in shared memory (<= 38 bf16)
constexpr int YS = 68;                  // row stride (floats) of the 64-wide exchange rows
constexpr int RECF = 16000;             // floats of the receive buffer (all senders)
constexpr int OWN_CW = 880, OWN_ROWS = 16;   // owner prefetch: Cw entries, window rows
constexpr long long kWait = 1ll << 31;

// shared-memory map (bytes)
constexpr int OB_HI = 0;                                   // [W^T (64 rows); S^T (64); X (Kw)] x FS, hi
constexpr int OB_LO = OB_HI + (128 + KWM) * FSM * 2;       // the same, lo
constexpr int OR_HI = OB_LO + (128 + KWM) * FSM * 2;       // R (64 rows) x FS
constexpr int OR_LO = OR_HI + 64 * FSM * 2;
constexpr int DYT = KWM * 64 * 2;
constexpr int ODY = OR_LO + 64 * FSM * 2;                  // scaled dY, hi and lo: [Kw][64] each
constexpr int OREC = ODY + 2 * DYT;                        // partials received from the cluster
constexpr int ODYF = OREC + RECF * 4;                      // dY fp32 [Kw][YS]
constexpr int ORAW = ODYF + KWM * YS * 4;                  // raw rows: 64 queries, then Kw keys
constexpr int OVEC = ORAW + (64 + KWM) * RAWB;             // per-chunk gate vectors, by parity
constexpr int VECF = 296;
constexpr int OOWN = OVEC + 2 * VECF * 4;                  // owned rows' Cw, gamma, v (bf16)
constexpr int OOWN_G = OOWN + OWN_CW * 4;
constexpr int OOWN_V = OOWN_G + OWN_ROWS * 4;
constexpr int OTAB = OOWN_V + OWN_ROWS * 128;              // monomial table of the slice
constexpr int SMEM_BYTES = OTAB + FSM * 4;
static_assert(SMEM_BYTES + 1024 <= 227 * 1024, "shared memory map exceeds a CTA's limit");
static_assert(OREC % 16 == 0 && ODYF % 16 == 0 && ORAW % 16 == 0 && OVEC % 16 == 0 && OOWN_V % 16 == 0,
              "16-byte alignment");

// inside a gate-vector buffer
constexpr int V_BT = 0, V_DT = 64, V_CS = 128, V_CW = 208, V_ABD = 288;

// TMEM columns
constexpr uint32_t T_G1 = 0;     // [RW | RS | RX], M = 64 layout
constexpr uint32_t T_XW = 224;   // X W^, M = 128 layout
constexpr uint32_t T_D1 = 0, T_D2 = 96;        // state corrections (M = 64, transposed)
constexpr uint32_t T_W = 288, T_S = 384;       // fp32 masters W^T, S^T (M = 64, transposed)

struct P1 {
  int nc, fs, kwp, yr, xr, nchunks;
  int blockf;   // floats of one sender's block in the receive buffer
  int own_pf;   // the owned rows' Cw, gamma, v fit the prefetch buffers
};

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(cta));
  return r;
}
__device__ __forceinline__ void st_peer4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 8 consecutive fp32 values -> bf16 hi and lo chunks (16 bytes each) at off
__device__ __forceinline__ void put8(uint8_t* hi, uint8_t* lo, uint32_t off, const float* v) {
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

__device__ __forceinline__ void sync_mma() {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// D = A B over K in split bf16 (three products), one thread.  Descriptor
// strides: K-major operands lbo = 128, sbo = row-group stride, K step 256 B;
// MN-major lbo = k-group stride, sbo = 128, K step two k-groups.
struct Opnd {
  uint32_t hi, lo;   // shared addresses
  uint32_t lbo, sbo, kstep;
};
__device__ __forceinline__ Opnd kmajor(const uint8_t* hi, const uint8_t* lo, int rgs) {
  return Opnd{tc::smem_u32(hi), tc::smem_u32(lo), 128u, (uint32_t)rgs, 256u};
}
__device__ __forceinline__ Opnd mnmajor(const uint8_t* hi, const uint8_t* lo, int kgs) {
  return Opnd{tc::smem_u32(hi), tc::smem_u32(lo), (uint32_t)kgs, 128u, (uint32_t)(2 * kgs)};
}
__device__ __forceinline__ void mma_split(uint32_t d, const Opnd& a, const Opnd& b, uint32_t idesc, int K) {
  const uint32_t as[3] = {a.hi, a.hi, a.lo}, bs[3] = {b.hi, b.lo, b.hi};
  for (int p = 0; p < 3; ++p) {
    uint64_t ad = tc::sdesc(as[p], a.lbo, a.sbo), bd = tc::sdesc(bs[p], b.lbo, b.sbo);
    for (int ks = 0; ks < K / 16; ++ks) {
      tc::mma_f16(d, ad, bd, idesc, (p > 0 || ks > 0) ? 1u : 0u);
      ad += a.kstep >> 4;
      bd += b.kstep >> 4;
    }
  }
}

// Bounded wait for the MMA group just committed; a timeout is recorded and
// turns this CTA's MMA issue off for the rest of the call.
__device__ __forceinline__ bool wait_group(uint64_t* bar, uint32_t& phase, bool ok, int* status) {
  bool good = true;
  if (ok) good = tc::mbar_wait(bar, phase, kWait);
  phase ^= 1;
  const bool bad = __syncthreads_or(!good);
  if (bad && threadIdx.x == 0) atomicExch(status, ATLAS_ERR_TIMEOUT);
  tc::fence_after_sync();
  return ok && !bad;
}

// key row l of the unit (window-cache rows first): its bf16 value row and
// its Omega weight (nullptr: weight 1), in the call's inputs
__device__ __forceinline__ const uint16_t* v_row(const Geom& g, const GenericIO& io, int u, int l) {
  return l < g.n_prev ? (const uint16_t*)io.win_v + ((size_t)u * (g.c - 1) + (g.c - 1 - g.n_prev + l)) * g.d_v
                      : (const uint16_t*)io.v + ((size_t)u * g.T + (l - g.n_prev)) * g.d_v;
}
__device__ __forceinline__ const float* gamma_ptr(const Geom& g, const GenericIO& io, int u, int l) {
  if (l < g.n_prev)
    return io.win_gamma ? io.win_gamma + (size_t)u * (g.c - 1) + (g.c - 1 - g.n_prev + l) : nullptr;
  return io.gamma ? io.gamma + (size_t)u * g.T + (l - g.n_prev) : nullptr;
}

}  // namespace

namespace {

// cp.async of chunk n's raw query and window-key rows (bf16) and its gate
// vectors; entries past the chunk (t >= C, i >= nw) of the vectors are zero.
__device__ void prefetch_chunk(const Geom& g, const GenericIO& io, const float* coef, const P1& pp, int u, int n,
                               uint16_t* raw, float* vec) {
  const Chunk ch = dual1_chunk_at(g, n * g.C);
  const int dk = g.d_k, pieces = dk / 8, C = g.C, Kw = g.Kw;
  for (int e = threadIdx.x; e < C * pieces; e += NT) {
    const int t = e / pieces, pc = e % pieces;
    cp16(raw + t * (RAWB / 2) + pc * 8, (const uint16_t*)io.q + ((size_t)u * g.T + ch.s + t) * dk + pc * 8);
  }
  for (int e = threadIdx.x; e < ch.nw * pieces; e += NT) {
    const int i = e / pieces, pc = e % pieces;
    const int l = ch.lo + g.n_prev + i;   // key row of the unit, window-cache rows first
    const uint16_t* src =
        l < g.n_prev ? (const uint16_t*)io.win_k + ((size_t)u * (g.c - 1) + (g.c - 1 - g.n_prev + l)) * dk
                     : (const uint16_t*)io.k + ((size_t)u * g.T + (l - g.n_prev)) * dk;
    cp16(raw + (64 + i) * (RAWB / 2) + pc * 8, src + pc * 8);
  }
  const float* cb = coef + ((size_t)u * pp.nchunks + n) * dual1_coef_floats(g);
  const float* cse = cb + (size_t)C * Kw;
  const float* cwe = cse + Kw;
  const float* Bt = cwe + Kw;
  const float* Dt = Bt + C;
  const float* ABD = Dt + C;
  float* vb = vec + (n & 1) * VECF;
  for (int e = threadIdx.x; e < 64; e += NT) {
    cp4(vb + V_BT + e, e < C ? Bt + e : cb, e < C);
    cp4(vb + V_DT + e, e < C ? Dt + e : cb, e < C);
  }
  for (int e = threadIdx.x; e < KWM; e += NT) {
    cp4(vb + V_CS + e, e < ch.nw ? cse + e : cb, e < ch.nw);
    cp4(vb + V_CW + e, e < ch.nw ? cwe + e : cb, e < ch.nw);
  }
  if (threadIdx.x < 3) cp4(vb + V_ABD + threadIdx.x, ABD + threadIdx.x, true);
  cp_commit();
}

// cp.async of what the owner of rows t in [rank YR, +YR) and window rows
// i in [rank XR, +XR) reads in chunk n: Cw_t[i], gamma_i, v_i (bf16).  An
// empty group when they do not fit (the owner then reads them directly).
__device__ void prefetch_owner(const Geom& g, const GenericIO& io, const float* coef, const P1& pp, int u, int n,
                               int rank, float* ocw, float* og, uint16_t* ov) {
  if (pp.own_pf) {
    const Chunk ch = dual1_chunk_at(g, n * g.C);
    const float* Cw = coef + ((size_t)u * pp.nchunks + n) * dual1_coef_floats(g);
    const int Kw = g.Kw;
    for (int e = threadIdx.x; e < pp.yr * Kw; e += NT) {
      const int r = e / Kw, i = e % Kw, t = rank * pp.yr + r;
      const bool in = t < g.C && i < ch.nw;
      cp4(ocw + e, in ? Cw + (size_t)t * Kw + i : Cw, in);
    }
    const int pieces = g.d_v / 8;
    for (int e = threadIdx.x; e < pp.xr * pieces; e += NT) {
      const int r = e / pieces, pc = e % pieces, i = rank * pp.xr + r;
      if (i < ch.nw) cp16(ov + r * 64 + pc * 8, v_row(g, io, u, ch.lo + g.n_prev + i) + pc * 8);
    }
    for (int r = threadIdx.x; r < pp.xr; r += NT) {
      const int i = rank * pp.xr + r;
      const float* gp = i < ch.nw ? gamma_ptr(g, io, u, ch.lo + g.n_prev + i) : nullptr;
      if (gp) cp4(og + r, gp, true);
      else og[r] = 1.f;
    }
  }
  cp_commit();
}

// The slice's query rows (R, 64 x FS) and window rows (X, Kw x FS) of the
// monomial map, split bf16, from the raw rows x' = [x, 1, 0]: feature f is
// s_f x'_a x'_b with (a, b, s_f = 1 or 1/2) from the slice's table.  Rows
// vary fastest across threads: the 16-byte stores of a warp then fall in
// distinct banks.
__device__ void generate_tiles(const Geom& g, const Chunk& ch, const P1& pp, int rgs, const uint16_t* raw,
                               const uint32_t* tab, uint8_t* r_hi, uint8_t* r_lo, uint8_t* x_hi, uint8_t* x_lo) {
  const int nch = pp.fs / 8, rows = 64 + pp.kwp;
  for (int e = threadIdx.x; e < rows * nch; e += NT) {
    const int r = e % rows, c8 = (e / rows) * 8;
    const bool isq = r < 64;
    const int i = r - 64;
    const bool valid = isq ? r < g.C : i < ch.nw;
    const uint16_t* xr = raw + r * (RAWB / 2);
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t t = tab[c8 + k];
      const float p = tc::bf2f(xr[t & 255u]) * tc::bf2f(xr[(t >> 8) & 255u]);
      v[k] = valid ? ((t >> 16) ? 0.5f * p : p) : 0.f;
    }
    if (isq) put8(r_hi, r_lo, tc::core_offset(r, c8, rgs), v);
    else put8(x_hi, x_lo, tc::core_offset(i, c8, rgs), v);
  }
}

// dY (fp32 rows) times a per-row scale -> the split MN-major operand tile
__device__ void scale_dy(const float* dyf, const float* sc, int kwp, uint8_t* hi, uint8_t* lo) {
  for (int e = threadIdx.x; e < kwp * 8; e += NT) {
    const int i = e % kwp, c8 = (e / kwp) * 8;
    const float4 v0 = *reinterpret_cast<const float4*>(dyf + i * YS + c8);
    const float4 v1 = *reinterpret_cast<const float4*>(dyf + i * YS + c8 + 4);
    const float s = sc[i];
    const float a[8] = {s * v0.x, s * v0.y, s * v0.z, s * v0.w, s * v1.x, s * v1.y, s * v1.z, s * v1.w};
    put8(hi, lo, tc::core_offset(i, c8, 1024), a);
  }
}

}  // namespace

__global__ void __launch_bounds__(NT, 1) k_dual1_tc(Geom g, Work w, GenericIO io, const float* coef, P1 pp,
                                                     int fbuf) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase_s;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int q4 = warp & 3, hw = warp >> 2;        // TMEM sub-partition, column half
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const uint32_t rank = cta_rank();
  const int u = blockIdx.y, NC = pp.nc, FS = pp.fs, KWP = pp.kwp, YR = pp.yr, XR = pp.xr;
  const int rgs = (FS / 8) * 128, f0 = (int)rank * FS, dv = g.d_v, dk = g.d_k, C = g.C;
  uint8_t* b_hi = sm + OB_HI;
  uint8_t* b_lo = sm + OB_LO;
  uint8_t* x_hi = b_hi + 16 * rgs;   // X starts at row 128 of the B tile
  uint8_t* x_lo = b_lo + 16 * rgs;
  uint8_t* r_hi = sm + OR_HI;
  uint8_t* r_lo = sm + OR_LO;
  uint8_t* d_hi = sm + ODY;
  uint8_t* d_lo = d_hi + DYT;
  float* rec = reinterpret_cast<float*>(sm + OREC);
  float* dyf = reinterpret_cast<float*>(sm + ODYF);
  uint16_t* raw = reinterpret_cast<uint16_t*>(sm + ORAW);
  float* vec = reinterpret_cast<float*>(sm + OVEC);
  float* ocw = reinterpret_cast<float*>(sm + OOWN);
  float* og = reinterpret_cast<float*>(sm + OOWN_G);
  uint16_t* ov = reinterpret_cast<uint16_t*>(sm + OOWN_V);
  uint32_t* tab = reinterpret_cast<uint32_t*>(sm + OTAB);
  float* mine = rec + rank * pp.blockf;            // this CTA's own block: the owned rows' sums land here
  const int oRX = YR * YS, oXW = YR * YS + YR * (KWP + 4);   // regions inside a sender's block

  if (warp == 0) tc::tmem_alloc(&tbase_s, 512);
  if (tid == 0) tc::mbar_init(&bar, 1);
  // monomial table of the slice: feature f = s_f x'_a x'_b over x' = [x, 1, 0]
  for (int fl = tid; fl < FS; fl += NT) {
    const int f = f0 + fl;
    int a = dk + 1, b = dk + 1, half = 0;   // padding: 0 * 0
    if (f < g.F) {
      if (g.p == 1) {
        a = f;
        b = dk;
      } else if (f == 0) {
        a = dk;
        b = dk;
      } else if (f <= dk) {
        a = f - 1;
        b = dk;
      } else {   // x_i x_j / 2, i <= j, lexicographic
        int r = f - 1 - dk, i = 0;
        while (r >= dk - i) {
          r -= dk - i;
          ++i;
        }
        a = i;
        b = i + r;
        half = 1;
      }
    }
    tab[fl] = (uint32_t)a | ((uint32_t)b << 8) | ((uint32_t)half << 16);
  }
  for (int r = tid; r < 64 + KWM; r += NT) {
    raw[r * (RAWB / 2) + dk] = 0x3F80;   // bf16 1.0
    raw[r * (RAWB / 2) + dk + 1] = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tbase_s;

  // the call's initial W, S slice -> fp32 masters (transposed) and operand copies
  {
    const float* Wg = w.Wst[0][0] + (size_t)u * g.F * dv;
    const float* Sg = w.Sst[0][0] + (size_t)u * g.F * dv;
    const int j = 16 * q4 + (lane & 15);
    for (int cb = 32 * hw; cb < FS; cb += 64) {
      const int fc = cb + 16 * (lane >> 4);
      float vw[16], vs[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int f = f0 + fc + k;
        const bool in = fc + k < FS && f < g.F && j < dv;
        vw[k] = in ? Wg[(size_t)f * dv + j] : 0.f;
        vs[k] = in ? Sg[(size_t)f * dv + j] : 0.f;
      }
      tc::tmem_st16_x2(tb + lane_base + T_W + cb, vw);
      tc::tmem_st16_x2(tb + lane_base + T_S + cb, vs);
      if (fc < FS) {
        put8(b_hi, b_lo, tc::core_offset(j, fc, rgs), vw);
        put8(b_hi, b_lo, tc::core_offset(j, fc + 8, rgs), vw + 8);
        put8(b_hi, b_lo, tc::core_offset(64 + j, fc, rgs), vs);
        put8(b_hi, b_lo, tc::core_offset(64 + j, fc + 8, rgs), vs + 8);
      }
    }
    tc::tmem_st_wait();
  }
  // cp.async groups in commit order: chunk(0), owner(0), then per chunk n:
  // chunk(n + 1) during the first MMA group, owner(n + 1) after barrier B2
  prefetch_chunk(g, io, coef, pp, u, 0, raw, vec);
  prefetch_owner(g, io, coef, pp, u, 0, (int)rank, ocw, og, ov);
  tc::fence_before_sync();
  cluster_barrier();   // every CTA of the cluster runs: its shared memory takes peer stores from here on
  tc::fence_after_sync();

  bool ok = true;
  uint32_t phase = 0;
  for (int n = 0; n < pp.nchunks; ++n) {
    const Chunk ch = dual1_chunk_at(g, n * C);
    const float* vb = vec + (n & 1) * VECF;
    const bool more = n + 1 < pp.nchunks;
    cp_wait<1>();   // chunk(n) has landed; owner(n) may still be in flight
    __syncthreads();
    generate_tiles(g, ch, pp, rgs, raw, tab, r_hi, r_lo, x_hi, x_lo);

    // 2. partial products of the slice; the next chunk's rows load meanwhile
    sync_mma();   // also: every read of the raw rows is done
    if (tid == 0 && ok) {
      mma_split(tb + T_G1, kmajor(r_hi, r_lo, rgs), kmajor(b_hi, b_lo, rgs), tc::idesc_f16(64, 128 + KWP, 1, 0, 0),
                FS);
      mma_split(tb + T_XW, kmajor(x_hi, x_lo, rgs), kmajor(b_hi, b_lo, rgs), tc::idesc_f16(128, 64, 1, 0, 0), FS);
      tc::mma_commit(&bar);
    }
    if (more) prefetch_chunk(g, io, coef, pp, u, n + 1, raw, vec);
    ok = wait_group(&bar, phase, ok, w.status);

    // 3. partials to their owners: rows t of Yp = B_t RW + D_t RS and of R X^T
    //    (owner t / YR), rows i of X W^ (owner i / XR)
    {
      const uint32_t blk = tc::smem_u32(rec) + rank * (uint32_t)pp.blockf * 4u;   // this sender's block
      const int t = 16 * q4 + (lane & 15), owner = t / YR, tr = t % YR;
      if (hw == 0) {
        const float bt = vb[V_BT + t], dt = vb[V_DT + t];
        for (int cb = 0; cb < 64; cb += 32) {
          float a[16], s[16];
          tc::tmem_ld16_x2(tb + lane_base + T_G1 + cb, a);
          tc::tmem_ld16_x2(tb + lane_base + T_G1 + 64 + cb, s);
          tc::tmem_ld_wait();
          const int j0 = cb + 16 * (lane >> 4);
          const uint32_t dst = peer_addr(blk + (uint32_t)(tr * YS + j0) * 4u, owner);
#pragma unroll
          for (int k = 0; k < 16; k += 4)
            st_peer4(dst + 4u * k, bt * a[k] + dt * s[k], bt * a[k + 1] + dt * s[k + 1], bt * a[k + 2] + dt * s[k + 2],
                     bt * a[k + 3] + dt * s[k + 3]);
        }
      } else {
        for (int cb = 0; cb < KWP; cb += 32) {
          float a[16];
          tc::tmem_ld16_x2(tb + lane_base + T_G1 + 128 + cb, a);
          tc::tmem_ld_wait();
          const int i0 = cb + 16 * (lane >> 4);
          if (i0 < KWP) {
            const uint32_t dst = peer_addr(blk + (uint32_t)(oRX + tr * (KWP + 4) + i0) * 4u, owner);
#pragma unroll
            for (int k = 0; k < 16; k += 4) st_peer4(dst + 4u * k, a[k], a[k + 1], a[k + 2], a[k + 3]);
          }
        }
      }
      if (32 * q4 < KWP) {   // X W^ rows in the M = 128 lanes: i = 32 q4 + lane, columns [32 hw, 32 hw + 32)
        float a[32];
        tc::tmem_ld16(tb + lane_base + T_XW + 32 * hw, a);
        tc::tmem_ld16(tb + lane_base + T_XW + 32 * hw + 16, a + 16);
        tc::tmem_ld_wait();
        const int i = 32 * q4 + lane;
        if (i < KWP) {
          const uint32_t dst = peer_addr(blk + (uint32_t)(oXW + (i % XR) * YS + 32 * hw) * 4u, i / XR);
#pragma unroll
          for (int k = 0; k < 32; k += 4) st_peer4(dst + 4u * k, a[k], a[k + 1], a[k + 2], a[k + 3]);
        }
      }
    }
    if (more) cp_wait<1>();   // owner(n) has landed; chunk(n + 1) may still be in flight
    else cp_wait<0>();
    tc::fence_before_sync();
    cluster_barrier();   // B1: every partial has arrived
    tc::fence_after_sync();

    // 4. the owned rows: sums over the NC senders in rank order
    {
      const float* Cwg = coef + ((size_t)u * pp.nchunks + n) * dual1_coef_floats(g);
      for (int e = tid; e < YR * 64; e += NT) {
        const int r = e >> 6, j = e & 63;
        if ((int)rank * YR + r >= 64) break;
        float s = 0.f;
        for (int src = 0; src < NC; ++src) s += rec[src * pp.blockf + r * YS + j];
        mine[r * YS + j] = s;
      }
      for (int e = tid; e < YR * KWP; e += NT) {
        const int r = e / KWP, i = e % KWP, t = (int)rank * YR + r;
        if (t >= 64) break;
        float s = 0.f;
        for (int src = 0; src < NC; ++src) s += rec[src * pp.blockf + oRX + r * (KWP + 4) + i];
        float cw = 0.f;
        if (t < C && i < ch.nw) cw = pp.own_pf ? ocw[r * g.Kw + i] : Cwg[(size_t)t * g.Kw + i];
        mine[oRX + r * (KWP + 4) + i] = cw * s;
      }
      for (int e = tid; e < XR * 16; e += NT) {
        const int r = e >> 4, j0 = (e & 15) * 4, i = (int)rank * XR + r;
        if (i >= KWP) break;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (i < ch.nw) {
          const int l = ch.lo + g.n_prev + i;
          float gm = 1.f;
          if (pp.own_pf) {
            gm = og[r];
          } else {
            const float* gp = gamma_ptr(g, io, u, l);
            if (gp) gm = *gp;
          }
          const uint16_t* vr = pp.own_pf ? ov + r * 64 : v_row(g, io, u, l);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float s = 0.f;
            for (int src = 0; src < NC; ++src) s += rec[src * pp.blockf + oXW + r * YS + j0 + k];
            if (j0 + k < dv) d[k] = 2.f * gm * (s - tc::bf2f(vr[j0 + k]));
          }
        }
        const uint32_t loc = tc::smem_u32(dyf + i * YS + j0);
        for (int p = 0; p < NC; ++p) st_peer4(peer_addr(loc, p), d[0], d[1], d[2], d[3]);
      }
    }
    tc::fence_before_sync();
    cluster_barrier();   // B2: every dy row has arrived
    tc::fence_after_sync();
    if (more) prefetch_owner(g, io, coef, pp, u, n + 1, (int)rank, ocw, og, ov);

    // 5. chunk-end corrections on the tensor cores: (cs_e dY)^T X, then
    //    (cw_e dY)^T X through the same operand tile; the owned rows' read-out
    //    runs while the first one does
    scale_dy(dyf, vb + V_CS, KWP, d_hi, d_lo);
    sync_mma();
    const uint32_t ids = tc::idesc_f16(64, FS, 1, 1, 1);
    if (tid == 0 && ok) {
      mma_split(tb + T_D1, mnmajor(d_hi, d_lo, 1024), mnmajor(x_hi, x_lo, rgs), ids, KWP);
      tc::mma_commit(&bar);
    }
    for (int e = tid; e < YR * 64; e += NT) {
      const int r = e >> 6, j = e & 63, t = (int)rank * YR + r;
      if (t >= C) break;
      if (j >= dv) continue;
      const float* m = mine + oRX + r * (KWP + 4);
      float acc = mine[r * YS + j];
      for (int i = 0; i < KWP; ++i) acc -= m[i] * dyf[i * YS + j];
      io.y[((size_t)u * g.T + ch.s + t) * dv + j] = acc;
    }
    ok = wait_group(&bar, phase, ok, w.status);
    scale_dy(dyf, vb + V_CW, KWP, d_hi, d_lo);
    sync_mma();
    if (tid == 0 && ok) {
      mma_split(tb + T_D2, mnmajor(d_hi, d_lo, 1024), mnmajor(x_hi, x_lo, rgs), ids, KWP);
      tc::mma_commit(&bar);
    }
    ok = wait_group(&bar, phase, ok, w.status);

    // 6. chunk-end state of the slice
    {
      const float Ae = vb[V_ABD], Be = vb[V_ABD + 1], De = vb[V_ABD + 2];
      const int j = 16 * q4 + (lane & 15);
      for (int cb = 32 * hw; cb < FS; cb += 64) {
        float d1[16], d2[16], wv[16], sv[16];
        tc::tmem_ld16_x2(tb + lane_base + T_D1 + cb, d1);
        tc::tmem_ld16_x2(tb + lane_base + T_D2 + cb, d2);
        tc::tmem_ld16_x2(tb + lane_base + T_W + cb, wv);
        tc::tmem_ld16_x2(tb + lane_base + T_S + cb, sv);
        tc::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float s0 = sv[k];
          sv[k] = Ae * s0 - d1[k];
          wv[k] = Be * wv[k] + De * s0 - d2[k];
        }
        tc::tmem_st16_x2(tb + lane_base + T_W + cb, wv);
        tc::tmem_st16_x2(tb + lane_base + T_S + cb, sv);
        const int fc = cb + 16 * (lane >> 4);
        if (fc < FS) {
          put8(b_hi, b_lo, tc::core_offset(j, fc, rgs), wv);
          put8(b_hi, b_lo, tc::core_offset(j, fc + 8, rgs), wv + 8);
          put8(b_hi, b_lo, tc::core_offset(64 + j, fc, rgs), sv);
          put8(b_hi, b_lo, tc::core_offset(64 + j, fc + 8, rgs), sv + 8);
        }
      }
      tc::tmem_st_wait();
    }
  }

  // the call's final W, S slice
  {
    float* Wg = w.Wst[fbuf][0] + (size_t)u * g.F * dv;
    float* Sg = w.Sst[fbuf][0] + (size_t)u * g.F * dv;
    const int j = 16 * q4 + (lane & 15);
    for (int cb = 32 * hw; cb < FS; cb += 64) {
      float wv[16], sv[16];
      tc::tmem_ld16_x2(tb + lane_base + T_W + cb, wv);
      tc::tmem_ld16_x2(tb + lane_base + T_S + cb, sv);
      tc::tmem_ld_wait();
      const int fc = cb + 16 * (lane >> 4);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int f = f0 + fc + k;
        if (fc + k < FS && f < g.F && j < dv) {
          Wg[(size_t)f * dv + j] = wv[k];
          Sg[(size_t)f * dv + j] = sv[k];
        }
      }
    }
  }
  tc::fence_before_sync();
  cluster_barrier();   // no peer store into this CTA's shared memory is left in flight
  if (warp == 0) tc::tmem_dealloc(tb, 512);
}

namespace {

P1 plan(const Geom& g) {
  P1 p;
  p.nc = (g.F + FSM - 1) / FSM;
  if (p.nc < 1) p.nc = 1;
  p.fs = ((g.F + p.nc - 1) / p.nc + 15) / 16 * 16;
  p.kwp = (g.Kw + 15) / 16 * 16;
  p.yr = (64 + p.nc - 1) / p.nc;
  p.xr = (p.kwp + p.nc - 1) / p.nc;
  p.nchunks = g.T / g.C;
  p.blockf = p.yr * YS + p.yr * (p.kwp + 4) + p.xr * YS;
  p.own_pf = p.yr * g.Kw <= OWN_CW && p.xr <= OWN_ROWS;
  return p;
}

}  // namespace

bool dual1_tc_supported(const Geom& g) {
  if (!(g.depth == 1 && g.ns_iters == 0 && g.update == ATLAS_UPDATE_PER_TOKEN && g.qkv_dtype == ATLAS_BF16 &&
        g.proj_dim == 0 && (g.p == 1 || g.p == 2)))
    return false;
  if (g.d_k % 8 || g.d_k > 32 || g.d_v % 8 || g.d_v > 64 || g.C > 64 || g.Kw > KWM || g.F > 8 * FSM) return false;
  const P1 p = plan(g);
  return p.nc <= 8 && p.fs <= FSM && p.nc * p.blockf <= RECF;
}

bool dual1_tc_inputs_ok(const GenericIO& io) {
  // 16-byte copies of the raw key, query and value rows
  return ((uintptr_t)io.q % 16 == 0) && ((uintptr_t)io.k % 16 == 0) && ((uintptr_t)io.v % 16 == 0) &&
         ((uintptr_t)io.win_k % 16 == 0) && ((uintptr_t)io.win_v % 16 == 0);
}

cudaError_t dual1_tc_launch(const Geom& g, const Work& w, const GenericIO& io, const float* coef, int fbuf,
                            cudaStream_t st) {
  const P1 p = plan(g);
  cudaError_t e = cudaFuncSetAttribute(k_dual1_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nc, g.units, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = p.nc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_dual1_tc, g, w, io, coef, p, fbuf);
}

}  // namespace atlas
