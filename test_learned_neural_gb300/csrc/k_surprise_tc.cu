// Newton-Schulz on the windowed surprise, depth-2 memory: the chunk's
// read-out and chunk-end state on the tensor cores (the banded coefficient
// algebra around them stays in k_surprise.cu).  With L, R the window rows'
// factors of a matrix (W1: x_i and dz_i; W2: a_i and dy_i) and Mw_t, Ms_e
// the banded core-weight matrices (atlas-torch README, "Atlas Extensions":
// Newton-Schulz orthogonalises the surprise updates, eta outside it):
//
//   z_t = B_t r_t W1^ + D_t r_t S1^ - ((r_t L1^T) Mw1_t) R1,  aq_t = SiLU(z_t)
//   y_t = r_t + B_t aq_t W2^ + D_t aq_t S2^ - ((aq_t L2^T) Mw2_t) R2
//   S'  = A_e S^ - L^T (Ms_e R),   W' = B_e W^ + D_e S^ - L^T (Mw_e R)
//
// Over the chunk's tokens these are products with M = the chunk (64 rows);
// every product is split bf16 (hi hi' + hi lo' + lo hi', fp32 accumulation
// in TMEM), the precision of the fp32 path it replaces to about 2^-16.
//   k_surp_tc_g2:    one CTA per (16 tokens, unit), a unit's four in a
//                    cluster, once per read-out: G = R L1^T (or G' = aq L2^T,
//                    each CTA a quarter of K = hidden, the partials summed
//                    over distributed shared memory), the band mix G Mw_t
//                    (fp32, SIMT), split into the G2 tile the read-out reads
//                    (the same for all of a unit's column blocks)
//   k_surp_tc_z:     one CTA per (64 hidden columns, unit): [R W1^ | R S1^]
//                    and (G Mw1) R1; aq to global
//   k_surp_tc_y:     one CTA per (32 output columns, unit): [aq W2^ | aq S2^]
//                    over K = hidden in chunks of 64 and (G' Mw2) R2; y
//   k_surp_tc_state: one CTA per (128 x 128 tile of a matrix, unit): L^T [Ms_e R
//                    | Mw_e R] (N = 256) and the decayed chunk-start state
#include "atlas_common.cuh"
#include "tc.cuh"
#include "tc_split.cuh"

namespace atlas {
namespace {

constexpr int NT = 256;
constexpr int KWM = 80;   // window rows, padded to 16 (Kw <= 80)
constexpr long long kWait = 1ll << 31;

__host__ __device__ inline int kwp_of(const Geom& g) { return (g.Kw + 15) / 16 * 16; }

// B_t, D_t of the read-out of chunk row t (pre-update mode: the previous
// token's; the chunk-start state's for the first token)
__device__ __forceinline__ void readout_gates(const Geom& g, const Work& w, int u, int t, int Ct, float& bt,
                                              float& dt) {
  const int rr = (g.readout == ATLAS_READOUT_PRE ? -1 : 0) + t;
  const bool ok = rr >= 0 && t < Ct;
  bt = ok ? w.Bp[(size_t)u * g.C + rr] : (rr < 0 ? 1.f : 0.f);
  dt = ok ? w.Dp[(size_t)u * g.C + rr] : 0.f;
}

// 8 consecutive fp32 values of a row (16-byte aligned) or zeros
__device__ __forceinline__ void load8(const float* src, bool valid, float* v) {
  if (valid) {
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.f;
  }
}

// Items e < n of a staging loop, four per thread at a time: every global
// load of the four is issued before the shared-memory stores (load(e, v)
// fills 8 values, store(e, v) writes them).
template <class Load, class Store>
__device__ __forceinline__ void stage4(int n, Load load, Store store) {
  for (int e0 = threadIdx.x; e0 < n; e0 += 4 * NT) {
    float v[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (e0 + q * NT < n) load(e0 + q * NT, v[q]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (e0 + q * NT < n) store(e0 + q * NT, v[q]);
  }
}

// Items [0, n1) of one staging loop and [0, n2) of another, PER per thread
// (n1 + n2 <= PER NT): every global load of both is issued before the
// shared-memory stores.
template <int PER, class L1, class S1, class L2, class S2>
__device__ __forceinline__ void stage2(int n1, int n2, L1 load1, S1 store1, L2 load2, S2 store2) {
  float v[PER][8];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = threadIdx.x + q * NT;
    if (e < n1) load1(e, v[q]);
    else if (e < n1 + n2) load2(e - n1, v[q]);
  }
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = threadIdx.x + q * NT;
    if (e < n1) store1(e, v[q]);
    else if (e < n1 + n2) store2(e - n1, v[q]);
  }
}

// G (fp32, M = 64 accumulator lanes, TMEM columns [col, col + kwp)) -> rows
// of gf (stride kwp + 4)
__device__ __forceinline__ void tmem_rows64_to_smem(uint32_t taddr_col, int kwp, float* gf) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, q4 = warp & 3, hw = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int t = 16 * q4 + (lane & 15);
  for (int cb = 32 * hw; cb < kwp; cb += 64) {
    float v[16];
    tc::tmem_ld16_x2(taddr_col + lane_base + cb, v);
    tc::tmem_ld_wait();
    const int c0 = cb + 16 * (lane >> 4);
    if (c0 < kwp)
#pragma unroll
      for (int k = 0; k < 16; ++k) gf[t * (kwp + 4) + c0 + k] = v[k];
  }
}

// n floats from global src to shared dst + mis by asynchronous copies, all
// in flight at once (16-byte copies where both sides allow it); mis = src's
// float offset inside its 16-byte chunk, so dst + mis shares src's
// alignment.  Returns mis once every copy has landed (this thread's).
__device__ __forceinline__ int stage_async(float* dst, const float* src, int n) {
  const int mis = (int)((reinterpret_cast<uintptr_t>(src) >> 2) & 3);
  const int head = mis ? (4 - mis < n ? 4 - mis : n) : 0;   // floats before src's first 16-byte boundary
  const int nb = (n - head) / 4;                            // 16-byte chunks after them
  float* d = dst + mis;
  if (threadIdx.x < head)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(d + threadIdx.x)), "l"(src + threadIdx.x)
                 : "memory");
  for (int b = threadIdx.x; b < nb; b += NT)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(d + head + 4 * b)),
                 "l"(src + head + 4 * b)
                 : "memory");
  for (int e = head + 4 * nb + threadIdx.x; e < n; e += NT)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(d + e)), "l"(src + e) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  return mis;
}

// G2[t][j] = sum_i G[t][i] Mw_t[i][j] over the band |i - j| < c for rows
// t in [tb, te), split into the K-major A tile [t][j] (rgs); rows t >= Ct
// and columns j >= nw are zero.
// The tokens' band matrices (contiguous in global memory) are staged in
// groups of tokens through `stage` (cap floats, at least one token's Kw (2c -
// 1) + 3) by asynchronous copies, so the sums read shared memory.
__device__ __forceinline__ void band_mix(const Geom& g, const Chunk& ch, const float* gf, int kwp, const float* mw,
                                         float* stage, int cap, uint8_t* hi, uint8_t* lo, int rgs, int tb, int te) {
  const int Ct = ch.e - ch.s, band = 2 * g.c - 1, nq = kwp / 8, per = g.Kw * band;
  const int MWG = (cap - 3) / per < te - tb ? (cap - 3) / per : te - tb;
  for (int t0 = tb; t0 < te; t0 += MWG) {
    const int lim = (Ct < te ? Ct : te) - t0;   // rows of this group that have a band matrix
    const int nt = lim < MWG ? (lim > 0 ? lim : 0) : MWG;
    const int mis = stage_async(stage, mw + (size_t)t0 * per, nt * per);
    __syncthreads();
    for (int e = threadIdx.x; e < MWG * nq; e += NT) {
      const int tt = e % MWG, t = t0 + tt, j0 = (e / MWG) * 8;
      if (t >= te) continue;   // the last group may reach past the rows
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int j = j0 + k;
        float acc = 0.f;
        if (tt < nt && j < ch.nw) {
          const int i0 = j - g.c + 1 > 0 ? j - g.c + 1 : 0, i1 = j + g.c - 1 < ch.nw - 1 ? j + g.c - 1 : ch.nw - 1;
          const float* M = stage + mis + tt * per;
          for (int i = i0; i <= i1; ++i) acc += gf[t * (kwp + 4) + i] * M[i * band + (j - i + g.c - 1)];
        }
        v[k] = acc;
      }
      tcs::put8(hi, lo, tc::core_offset(t, j0, rgs), v);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ band products
// G2 = (A L^T) Mw_t for the rows t of one 16-token group of the chunk: the
// hidden read-out's (ro = 0: A = the queries R, L = L1 = x_i, K = F) or the
// output read-out's (ro = 1: A = aq, L = L2 = a_i, K = hidden in chunks of
// 64).  It does not depend on the read-out's output columns, so it is formed
// once per unit here and written split (hi, lo) in the read-out kernels'
// K-major tile layout, which they copy into shared memory as is.
// shared memory (bytes): A [64][FZ], L [KWM][FZ] (K-major, hi + lo; the
// output read-out uses their first 64 columns per K chunk), G fp32 [64][KWM
// + 4], the G2 tile hi + lo, then the band staging
constexpr int FZ = 128;   // max F
constexpr int AG_A = 0, AG_L = AG_A + 2 * 64 * FZ * 2, AG_GF = AG_L + 2 * KWM * FZ * 2,
              AG_G2 = AG_GF + 64 * (KWM + 4) * 4, AG_MW = AG_G2 + 2 * 64 * KWM * 2, CAP_G = 16384,
              SMEM_G = AG_MW + CAP_G * 4;
static_assert(SMEM_G + 1024 <= 227 * 1024, "k_surp_tc_g2 shared memory");
static_assert(CAP_G >= KWM * 31 + 3, "one token's band matrix (c <= 16) fits the staging");

// the unit's G2 tile of read-out ro in the scratch (hi, then lo)
__device__ __forceinline__ uint8_t* g2_tile(const Work& w, const SurpOff& so, int u, int ro, int kwp) {
  return reinterpret_cast<uint8_t*>(w.surp + (size_t)u * so.per_unit + so.g2 + (size_t)ro * 64 * kwp);
}

// A unit's four token-group CTAs form a cluster.  For the output read-out
// each takes a quarter of the K loop over the hidden columns, and the owner
// of rows [16 q, 16 q + 16) sums the four partial G' rows over distributed
// shared memory in rank order (the same sum on every run).
__device__ __forceinline__ void cluster_sync4() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer(const float* p, uint32_t rank) {
  uint32_t a, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(tc::smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return __uint_as_float(v);
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(NT, 1)
    k_surp_tc_g2(Geom g, Chunk ch, Work w, SurpOff so, int ro, const float* aq) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, tb = 16 * blockIdx.x, te = tb + 16, u = blockIdx.y;
  const int F = g.F, h = g.hidden, Ct = ch.e - ch.s, nw = ch.nw, kwp = kwp_of(g);
  const int rgsF = (F / 8) * 128, rgs64 = 8 * 128, rgsK = (kwp / 8) * 128;
  uint8_t* a_hi = sm + AG_A;
  uint8_t* a_lo = a_hi + 64 * FZ * 2;
  uint8_t* l_hi = sm + AG_L;
  uint8_t* l_lo = l_hi + KWM * FZ * 2;
  uint8_t* g2_hi = sm + AG_G2;
  uint8_t* g2_lo = g2_hi + 64 * KWM * 2;
  float* gf = reinterpret_cast<float*>(sm + AG_GF);
  if ((tid >> 5) == 0) tc::tmem_alloc(&tbase, 128);
  if (tid == 0) tc::mbar_init(&bar, 1);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tG = tbase;
  bool ok = true;
  uint32_t phase = 0;
  bool have = true;   // this CTA's TMEM holds a product
  if (ro == 0) {
    const float* Rg = w.R + ((size_t)u * g.T + ch.s) * F;
    const float* Xg = w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * F;
    stage2<(64 * 16 + KWM * 16 + NT - 1) / NT>(
        64 * (F / 8), kwp * (F / 8),
        [&](int e, float* v) { load8(Rg + (size_t)(e % 64) * F + (e / 64) * 8, e % 64 < Ct, v); },
        [&](int e, const float* v) { tcs::put8(a_hi, a_lo, tc::core_offset(e % 64, (e / 64) * 8, rgsF), v); },
        [&](int e, float* v) { load8(Xg + (size_t)(e % kwp) * F + (e / kwp) * 8, e % kwp < nw, v); },
        [&](int e, const float* v) { tcs::put8(l_hi, l_lo, tc::core_offset(e % kwp, (e / kwp) * 8, rgsF), v); });
    tcs::sync_for_mma();
    if (tid == 0)
      tcs::mma3(tG, tcs::kmajor(a_hi, a_lo, rgsF), tcs::kmajor(l_hi, l_lo, rgsF), tc::idesc_f16(64, kwp, 1, 0, 0), F,
                false);
    ok = tcs::commit_wait(&bar, phase, ok, kWait);
  } else {
    // G' = aq L2^T over K = hidden in chunks of 64; each chunk's loads in
    // flight together, the next chunk's during this chunk's product
    const float* AQg = aq + (size_t)u * g.C * h;
    const float* Ag = w.Aact + (size_t)u * g.Kw * h;
    constexpr int GPER = (64 * 8 + KWM * 8 + NT - 1) / NT;
    const int ng = 64 * 8 + kwp * 8;
    auto g_load = [&](int e, int k0, float* v) {
      if (e < 512) load8(AQg + (size_t)(e % 64) * h + k0 + (e / 64) * 8, e % 64 < Ct, v);
      else load8(Ag + (size_t)((e - 512) % kwp) * h + k0 + ((e - 512) / kwp) * 8, (e - 512) % kwp < nw, v);
    };
    auto g_store = [&](int e, const float* v) {
      if (e < 512) tcs::put8(a_hi, a_lo, tc::core_offset(e % 64, (e / 64) * 8, rgs64), v);
      else tcs::put8(l_hi, l_lo, tc::core_offset((e - 512) % kwp, ((e - 512) / kwp) * 8, rgs64), v);
    };
    // this CTA's quarter of the 64-column chunks
    const int nch = h / 64, kb = (int)blockIdx.x * nch / 4 * 64, ke = ((int)blockIdx.x + 1) * nch / 4 * 64;
    float gv[GPER][8];
#pragma unroll
    for (int q = 0; q < GPER; ++q)
      if (kb < ke && tid + q * NT < ng) g_load(tid + q * NT, kb, gv[q]);
    for (int k0 = kb; k0 < ke; k0 += 64) {
#pragma unroll
      for (int q = 0; q < GPER; ++q)
        if (tid + q * NT < ng) g_store(tid + q * NT, gv[q]);
      tcs::sync_for_mma();
      if (tid == 0 && ok)
        tcs::mma3(tG, tcs::kmajor(a_hi, a_lo, rgs64), tcs::kmajor(l_hi, l_lo, rgs64), tc::idesc_f16(64, kwp, 1, 0, 0),
                  64, k0 > kb);
      if (k0 + 64 < ke) {
#pragma unroll
        for (int q = 0; q < GPER; ++q)
          if (tid + q * NT < ng) g_load(tid + q * NT, k0 + 64, gv[q]);
      }
      ok = tcs::commit_wait(&bar, phase, ok, kWait);   // the chunk's tiles are free again
    }
    have = kb < ke;
    if (!have) {
      // no chunk here: a zero partial
      for (int e = tid; e < 64 * (kwp + 4); e += NT) gf[e] = 0.f;
    }
  }
  if (have) tmem_rows64_to_smem(tG, kwp, gf);
  __syncthreads();
  if (ro == 1) {
    // G' rows [tb, te) = the four partials summed in rank order, written
    // over this CTA's own partial rows (no peer reads those)
    cluster_sync4();   // every partial is in its CTA's shared memory
    for (int e = tid; e < 16 * kwp; e += NT) {
      const int t = tb + e / kwp, i = e % kwp;
      const float* p = gf + t * (kwp + 4) + i;
      float acc = ld_peer(p, 0);
      for (int rk = 1; rk < 4; ++rk) acc += ld_peer(p, (uint32_t)rk);
      gf[t * (kwp + 4) + i] = acc;
    }
    cluster_sync4();   // every peer has read this CTA's rows
  }
  band_mix(g, ch, gf, kwp, w.surp + (size_t)u * so.per_unit + so.mwb + (size_t)ro * g.C * g.Kw * (2 * g.c - 1),
           reinterpret_cast<float*>(sm + AG_MW), CAP_G, g2_hi, g2_lo, rgsK, tb, te);
  // this group's two row groups of the hi and lo tiles to the scratch
  uint8_t* dst = g2_tile(w, so, u, ro, kwp);
  const int tile = 64 * kwp * 2, nb = 2 * rgsK / 16;
  for (int e = tid; e < 2 * nb; e += NT) {
    const int part = e / nb, off = (tb / 8) * rgsK + (e % nb) * 16;
    *reinterpret_cast<uint4*>(dst + part * tile + off) =
        *reinterpret_cast<const uint4*>((part ? g2_lo : g2_hi) + off);
  }
  if (!ok && tid == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if ((tid >> 5) == 0) tc::tmem_dealloc(tG, 128);
}

// the unit's G2 tile of read-out ro from the scratch into shared memory (hi,
// lo), by 16-byte asynchronous copies; waited for by the caller's
// cp.async.wait_group
__device__ __forceinline__ void g2_fetch(const Work& w, const SurpOff& so, int u, int ro, int kwp, uint8_t* hi,
                                         uint8_t* lo) {
  const uint8_t* src = g2_tile(w, so, u, ro, kwp);
  const int tile = 64 * kwp * 2, nb = tile / 16;
  for (int e = threadIdx.x; e < 2 * nb; e += NT) {
    const int part = e / nb, off = (e % nb) * 16;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32((part ? lo : hi) + off)),
                 "l"(src + part * tile + off)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// ------------------------------------------------------------ hidden read-out
// shared memory (bytes): R [64][F] (K-major), the W1 block and then the S1
// block [F][64] (MN-major, one buffer), DZ block [kwp][64] (MN-major), G2
// [64][kwp] (K-major), each hi + lo: 104 KB, two CTAs per SM
constexpr int AZ_R = 0, AZ_WS = AZ_R + 2 * 64 * FZ * 2, AZ_DZ = AZ_WS + 2 * FZ * 64 * 2,
              AZ_G2 = AZ_DZ + 2 * KWM * 64 * 2, SMEM_Z = AZ_G2 + 2 * 64 * KWM * 2;
static_assert(SMEM_Z + 1024 <= 227 * 1024, "k_surp_tc_z shared memory");

__global__ void __launch_bounds__(NT, 1) k_surp_tc_z(Geom g, Chunk ch, Work w, int buf, SurpOff so, float* aq) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, q4 = warp & 3, hw = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int jb = blockIdx.x * 64, u = blockIdx.y;
  const int F = g.F, h = g.hidden, Ct = ch.e - ch.s, nw = ch.nw, kwp = kwp_of(g);
  const int rgsF = (F / 8) * 128, rgsW = 8 * 128, rgsD = 8 * 128, rgsK = (kwp / 8) * 128;
  uint8_t* r_hi = sm + AZ_R;
  uint8_t* r_lo = r_hi + 64 * FZ * 2;
  uint8_t* ws_hi = sm + AZ_WS;
  uint8_t* ws_lo = ws_hi + FZ * 64 * 2;
  uint8_t* dz_hi = sm + AZ_DZ;
  uint8_t* dz_lo = dz_hi + KWM * 64 * 2;
  uint8_t* g2_hi = sm + AZ_G2;
  uint8_t* g2_lo = g2_hi + 64 * KWM * 2;

  if (warp == 0) tc::tmem_alloc(&tbase, 256);
  if (tid == 0) tc::mbar_init(&bar, 1);
  // operands: query features, the state blocks, dz_i, and the unit's G2 tile
  g2_fetch(w, so, u, 0, kwp, g2_hi, g2_lo);
  const float* Rg = w.R + ((size_t)u * g.T + ch.s) * F;
  const float* Wg = w.Wst[buf][0] + (size_t)u * F * h + jb;
  const float* Sg = w.Sst[buf][0] + (size_t)u * F * h + jb;
  const float* DZg = w.DZ + (size_t)u * g.Kw * h + jb;
  // staging rounds with every load of a round in flight at once: the W1
  // block with dz, then R; after the first products the S1 block
  auto ws_store = [&](int e, const float* v) {
    tcs::put8(ws_hi, ws_lo, tc::core_offset(e % F, (e / F) * 8, rgsW), v);
  };
  stage2<(FZ * 8 + KWM * 8 + NT - 1) / NT>(
      F * 8, kwp * 8, [&](int e, float* v) { load8(Wg + (size_t)(e % F) * h + (e / F) * 8, true, v); }, ws_store,
      [&](int e, float* v) { load8(DZg + (size_t)(e % kwp) * h + (e / kwp) * 8, e % kwp < nw, v); },
      [&](int e, const float* v) { tcs::put8(dz_hi, dz_lo, tc::core_offset(e % kwp, (e / kwp) * 8, rgsD), v); });
  stage4(
      64 * (F / 8), [&](int e, float* v) { load8(Rg + (size_t)(e % 64) * F + (e / 64) * 8, e % 64 < Ct, v); },
      [&](int e, float* v) { tcs::put8(r_hi, r_lo, tc::core_offset(e % 64, (e / 64) * 8, rgsF), v); });
  asm volatile("cp.async.wait_group 0;" ::: "memory");   // the G2 tile
  tcs::sync_for_mma();
  const uint32_t tb = tbase, tD1 = tb, tD3 = tb + 128;
  bool ok = true;
  uint32_t phase = 0;
  // R W1^ into columns 0-63, (G Mw1) R1 (N = 64); then R S1^ into 64-127
  if (tid == 0) {
    tcs::mma3(tD1, tcs::kmajor(r_hi, r_lo, rgsF), tcs::mnmajor(ws_hi, ws_lo, rgsW), tc::idesc_f16(64, 64, 1, 0, 1), F,
              false);
    tcs::mma3(tD3, tcs::kmajor(g2_hi, g2_lo, rgsK), tcs::mnmajor(dz_hi, dz_lo, rgsD), tc::idesc_f16(64, 64, 1, 0, 1),
              kwp, false);
  }
  {
    float sv[(FZ * 8 + NT - 1) / NT][8];   // the S1 block's loads fly while the products run
#pragma unroll
    for (int q = 0; q < (FZ * 8 + NT - 1) / NT; ++q) {
      const int e = tid + q * NT;
      if (e < F * 8) load8(Sg + (size_t)(e % F) * h + (e / F) * 8, true, sv[q]);
    }
    ok = tcs::commit_wait(&bar, phase, ok, kWait);   // the W1 block is free
#pragma unroll
    for (int q = 0; q < (FZ * 8 + NT - 1) / NT; ++q) {
      const int e = tid + q * NT;
      if (e < F * 8) ws_store(e, sv[q]);
    }
  }
  tcs::sync_for_mma();
  if (tid == 0 && ok)
    tcs::mma3(tD1 + 64, tcs::kmajor(r_hi, r_lo, rgsF), tcs::mnmajor(ws_hi, ws_lo, rgsW), tc::idesc_f16(64, 64, 1, 0, 1),
              F, false);
  ok = tcs::commit_wait(&bar, phase, ok, kWait);
  // z = B_t (R W1^) + D_t (R S1^) - (G Mw1) R1, aq = SiLU(z)
  {
    const int t = 16 * q4 + (lane & 15);
    float bt, dt;
    readout_gates(g, w, u, t, Ct, bt, dt);
    const int cb = 32 * hw;
    float a[16], s[16], d3[16];
    tc::tmem_ld16_x2(tD1 + lane_base + cb, a);
    tc::tmem_ld16_x2(tD1 + lane_base + 64 + cb, s);
    tc::tmem_ld16_x2(tD3 + lane_base + cb, d3);
    tc::tmem_ld_wait();
    const int c0 = cb + 16 * (lane >> 4);
    if (t < Ct) {
      float* o = aq + ((size_t)u * g.C + t) * h + jb + c0;
#pragma unroll
      for (int k = 0; k < 16; k += 4)
        *reinterpret_cast<float4*>(o + k) =
            make_float4(siluf_(bt * a[k] + dt * s[k] - d3[k]), siluf_(bt * a[k + 1] + dt * s[k + 1] - d3[k + 1]),
                        siluf_(bt * a[k + 2] + dt * s[k + 2] - d3[k + 2]),
                        siluf_(bt * a[k + 3] + dt * s[k + 3] - d3[k + 3]));
    }
  }
  if (!ok && tid == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 256);
}

// ------------------------------------------------------------ output read-out
// shared memory (bytes): per K chunk of 64 hidden columns aq [64][64]
// (K-major) and [W2 | S2] rows [64][64] (MN-major); then G2' [64][kwp]
// (K-major) and the DY block [kwp][32] (MN-major); each hi + lo
constexpr int AY_AQ = 0, AY_WS = AY_AQ + 2 * 64 * 64 * 2, AY_G2 = AY_WS + 2 * 64 * 64 * 2,
              AY_DY = AY_G2 + 2 * 64 * KWM * 2, SMEM_Y = AY_DY + 2 * KWM * 32 * 2;
static_assert(SMEM_Y + 1024 <= 227 * 1024, "k_surp_tc_y shared memory");

__global__ void __launch_bounds__(NT, 1) k_surp_tc_y(Geom g, Chunk ch, Work w, int buf, SurpOff so, const float* aq,
                                                      float* y) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, q4 = warp & 3, hw = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int kb = blockIdx.x * 32, u = blockIdx.y;
  const int h = g.hidden, d = g.d_v, F = g.F, Ct = ch.e - ch.s, nw = ch.nw, kwp = kwp_of(g);
  const int rgs64 = 8 * 128, rgs32 = 4 * 128, rgsK = (kwp / 8) * 128;
  uint8_t* aq_hi = sm + AY_AQ;
  uint8_t* aq_lo = aq_hi + 64 * 64 * 2;
  uint8_t* ws_hi = sm + AY_WS;
  uint8_t* ws_lo = ws_hi + 64 * 64 * 2;
  uint8_t* g2_hi = sm + AY_G2;
  uint8_t* g2_lo = g2_hi + 64 * KWM * 2;
  uint8_t* dy_hi = sm + AY_DY;
  uint8_t* dy_lo = dy_hi + KWM * 32 * 2;

  if (warp == 0) tc::tmem_alloc(&tbase, 128);
  if (tid == 0) tc::mbar_init(&bar, 1);
  g2_fetch(w, so, u, 1, kwp, g2_hi, g2_lo);   // the unit's G2' tile, waited for after the K loop
  const float* AQg = aq + (size_t)u * g.C * h;
  const float* Wg = w.Wst[buf][1] + (size_t)u * h * d + kb;
  const float* Sg = w.Sst[buf][1] + (size_t)u * h * d + kb;
  const float* DYg = w.DY + (size_t)u * g.Kw * d + kb;
  stage4(
      kwp * 4, [&](int e, float* v) { load8(DYg + (size_t)(e % kwp) * d + (e / kwp) * 8, e % kwp < nw, v); },
      [&](int e, float* v) { tcs::put8(dy_hi, dy_lo, tc::core_offset(e % kwp, (e / kwp) * 8, rgs32), v); });
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tbase, tD1 = tb, tD3 = tb + 64;
  bool ok = true;
  uint32_t phase = 0;
  // [aq W2^ | aq S2^] (N = 64), K = hidden in chunks of 64.  A chunk's two
  // tiles are items [0, 512) aq rows and [512, 1024) W2 / S2 rows, YPER per
  // thread: all of a chunk's loads are issued at once, the next chunk's
  // while this chunk's product runs.
  constexpr int YPER = (2 * 64 * 8 + NT - 1) / NT;
  const int ny = 2 * 64 * 8;
  auto y_load = [&](int e, int k0, float* v) {
    if (e < 512) {
      load8(AQg + (size_t)(e % 64) * h + k0 + (e / 64) * 8, e % 64 < Ct, v);
    } else {
      const int f = e - 512, c0 = (f / 64) * 8;   // columns 0-31: W2, 32-63: S2
      load8((c0 < 32 ? Wg : Sg) + (size_t)(k0 + f % 64) * d + (c0 & 31), true, v);
    }
  };
  auto y_store = [&](int e, const float* v) {
    if (e < 512) {
      tcs::put8(aq_hi, aq_lo, tc::core_offset(e % 64, (e / 64) * 8, rgs64), v);
    } else {
      const int f = e - 512;
      tcs::put8(ws_hi, ws_lo, tc::core_offset(f % 64, (f / 64) * 8, rgs64), v);
    }
  };
  float yv[YPER][8];
#pragma unroll
  for (int q = 0; q < YPER; ++q)
    if (tid + q * NT < ny) y_load(tid + q * NT, 0, yv[q]);
  for (int k0 = 0; k0 < h; k0 += 64) {
#pragma unroll
    for (int q = 0; q < YPER; ++q)
      if (tid + q * NT < ny) y_store(tid + q * NT, yv[q]);
    tcs::sync_for_mma();
    if (tid == 0 && ok)
      tcs::mma3(tD1, tcs::kmajor(aq_hi, aq_lo, rgs64), tcs::mnmajor(ws_hi, ws_lo, rgs64),
                tc::idesc_f16(64, 64, 1, 0, 1), 64, k0 > 0);
    if (k0 + 64 < h) {
#pragma unroll
      for (int q = 0; q < YPER; ++q)
        if (tid + q * NT < ny) y_load(tid + q * NT, k0 + 64, yv[q]);
    }
    ok = tcs::commit_wait(&bar, phase, ok, kWait);   // the chunk's tiles are free again
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");   // the G2' tile
  tcs::sync_for_mma();
  if (tid == 0 && ok)
    tcs::mma3(tD3, tcs::kmajor(g2_hi, g2_lo, rgsK), tcs::mnmajor(dy_hi, dy_lo, rgs32), tc::idesc_f16(64, 32, 1, 0, 1),
              kwp, false);
  ok = tcs::commit_wait(&bar, phase, ok, kWait);
  // y = r + B_t (aq W2^) + D_t (aq S2^) - (G' Mw2) R2
  if (hw == 0) {
    const int t = 16 * q4 + (lane & 15);
    float bt, dt;
    readout_gates(g, w, u, t, Ct, bt, dt);
    float a[16], s[16], d3[16];
    tc::tmem_ld16_x2(tD1 + lane_base, a);        // columns 0-31: aq W2^
    tc::tmem_ld16_x2(tD1 + lane_base + 32, s);   // columns 32-63: aq S2^
    tc::tmem_ld16_x2(tD3 + lane_base, d3);
    tc::tmem_ld_wait();
    const int c0 = 16 * (lane >> 4);
    if (t < Ct) {
      const size_t row = (size_t)u * g.T + ch.s + t;
      const float* rq = w.R + row * F + kb + c0;
      float* o = y + row * d + kb + c0;
#pragma unroll
      for (int k = 0; k < 16; k += 4) {
        const float4 r4 = *reinterpret_cast<const float4*>(rq + k);
        *reinterpret_cast<float4*>(o + k) =
            make_float4(r4.x + bt * a[k] + dt * s[k] - d3[k], r4.y + bt * a[k + 1] + dt * s[k + 1] - d3[k + 1],
                        r4.z + bt * a[k + 2] + dt * s[k + 2] - d3[k + 2],
                        r4.w + bt * a[k + 3] + dt * s[k + 3] - d3[k + 3]);
      }
    }
  }
  if (!ok && tid == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 128);
}

// -------------------------------------------------------------- chunk-end state
// shared memory (bytes): L^T tile [kwp][128] (MN-major A: rows i, columns the
// matrix rows of the tile), [Ms_e R | Mw_e R] tile [kwp][256] (MN-major B),
// each hi + lo
constexpr int AS_L = 0, AS_P = AS_L + 2 * KWM * 128 * 2, SMEM_S = AS_P + 2 * KWM * 256 * 2;
static_assert(SMEM_S + 1024 <= 227 * 1024, "k_surp_tc_state shared memory");

__global__ void __launch_bounds__(NT, 1) k_surp_tc_state(Geom g, Chunk ch, Work w, int buf, SurpOff so) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, q4 = warp & 3, hw = warp >> 2;
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int u = blockIdx.y, nw = ch.nw, kwp = kwp_of(g);
  // tile index -> (matrix, 128-row tile, 128-column block)
  int m = 0, tix = blockIdx.x;
  const int n0 = ((g.rows[0] + 127) / 128) * ((g.cols[0] + 127) / 128);
  if (tix >= n0) {
    m = 1;
    tix -= n0;
  }
  const int rows = g.rows[m], cols = g.cols[m], ncb = (cols + 127) / 128;
  const int r0 = (tix / ncb) * 128, c0 = (tix % ncb) * 128;
  const int rgsL = 16 * 128, rgsP = 32 * 128;
  uint8_t* l_hi = sm + AS_L;
  uint8_t* l_lo = l_hi + KWM * 128 * 2;
  uint8_t* p_hi = sm + AS_P;
  uint8_t* p_lo = p_hi + KWM * 256 * 2;
  if (warp == 0) tc::tmem_alloc(&tbase, 256);
  if (tid == 0) tc::mbar_init(&bar, 1);
  // L: the window rows' memory inputs (x_i for W1, a_i for W2), row width = rows
  const float* Lg = (m == 0) ? w.X + ((size_t)u * g.L + ch.lo + g.n_prev) * g.F : w.Aact + (size_t)u * g.Kw * g.hidden;
  const float* Pg = w.surp + (size_t)u * so.per_unit + so.rp + (size_t)m * 2 * g.Kw * so.maxcols;
  // both tiles' loads at once: items [0, 16 kwp) L rows, [16 kwp, 48 kwp)
  // the [Ms_e R | Mw_e R] rows (16 kwp is a multiple of NT: warp-uniform)
  constexpr int SPER = (KWM * 48 + NT - 1) / NT;
  const int nl = kwp * 16, ns = kwp * 48;
  {
    float sv[SPER][8];
#pragma unroll
    for (int q = 0; q < SPER; ++q) {
      const int e = tid + q * NT;
      if (e < nl) {
        const int i = e % kwp, a0 = (e / kwp) * 8;
        load8(Lg + (size_t)i * rows + r0 + a0, i < nw && r0 + a0 < rows, sv[q]);
      } else if (e < ns) {
        const int f = e - nl, i = f % kwp, b0 = (f / kwp) * 8, which = b0 >> 7, b = c0 + (b0 & 127);
        load8(Pg + ((size_t)which * g.Kw + i) * so.maxcols + b, i < nw && b < cols, sv[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < SPER; ++q) {
      const int e = tid + q * NT;
      if (e < nl) {
        tcs::put8(l_hi, l_lo, tc::core_offset(e % kwp, (e / kwp) * 8, rgsL), sv[q]);
      } else if (e < ns) {
        const int f = e - nl;
        tcs::put8(p_hi, p_lo, tc::core_offset(f % kwp, (f / kwp) * 8, rgsP), sv[q]);
      }
    }
  }
  tcs::sync_for_mma();
  const uint32_t tb = tbase;
  bool ok = true;
  uint32_t phase = 0;
  if (tid == 0)
    tcs::mma3(tb, tcs::mnmajor(l_hi, l_lo, rgsL), tcs::mnmajor(p_hi, p_lo, rgsP), tc::idesc_f16(128, 256, 1, 1, 1),
              kwp, false);
  // S' = A_e S^ - L^T (Ms_e R), W' = B_e W^ + D_e S^ - L^T (Mw_e R): this
  // thread's rows of S^ and W^ load while the product runs
  const int re = ch.e - 1 - ch.s;
  const float Ae = w.Ap[(size_t)u * g.C + re], Be = w.Bp[(size_t)u * g.C + re], De = w.Dp[(size_t)u * g.C + re];
  const int r = r0 + 32 * q4 + lane;   // M = 128: TMEM lane = tile row
  const size_t base = (size_t)u * rows * cols;
  float4 s4[4][4], w4[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = c0 + 64 * hw + 16 * j;
    if (r < rows && c < cols) {
      const size_t o = base + (size_t)r * cols + c;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        s4[j][k] = *reinterpret_cast<const float4*>(w.Sst[buf][m] + o + 4 * k);
        w4[j][k] = *reinterpret_cast<const float4*>(w.Wst[buf][m] + o + 4 * k);
      }
    }
  }
  ok = tcs::commit_wait(&bar, phase, ok, kWait);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int cb = 64 * hw + 16 * j;
    float ds[16], dw[16];
    tc::tmem_ld16(tb + lane_base + cb, ds);
    tc::tmem_ld16(tb + lane_base + 128 + cb, dw);
    tc::tmem_ld_wait();
    const int c = c0 + cb;
    if (r < rows && c < cols) {
      const size_t o = base + (size_t)r * cols + c;
      float* So = w.Sst[buf ^ 1][m] + o;
      float* Wo = w.Wst[buf ^ 1][m] + o;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 sb = s4[j][k], wb = w4[j][k];
        const float* dsk = ds + 4 * k;
        const float* dwk = dw + 4 * k;
        *reinterpret_cast<float4*>(So + 4 * k) =
            make_float4(Ae * sb.x - dsk[0], Ae * sb.y - dsk[1], Ae * sb.z - dsk[2], Ae * sb.w - dsk[3]);
        *reinterpret_cast<float4*>(Wo + 4 * k) =
            make_float4(Be * wb.x + De * sb.x - dwk[0], Be * wb.y + De * sb.y - dwk[1], Be * wb.z + De * sb.z - dwk[2],
                        Be * wb.w + De * sb.w - dwk[3]);
      }
    }
  }
  if (!ok && tid == 0) atomicExch(w.status, ATLAS_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 256);
}

}  // namespace

bool surprise_tc_supported(const Geom& g) {
  if (g.depth != 2 || g.ns_iters <= 0 || g.ns_target != ATLAS_NS_SURPRISE) return false;
  if (g.F % 16 || g.F > FZ || g.hidden % 64 || g.d_v % 32 || g.F < g.d_v) return false;
  if (g.F != g.d_v) return false;   // the residual read-out adds the query (F = d_v)
  if (g.C > 64 || g.Kw > KWM || g.c > 16) return false;
  if (g.rows[0] % 16 || g.rows[1] % 16 || g.cols[0] % 16 || g.cols[1] % 16) return false;
  // 16-byte loads of the Ms_e R, Mw_e R rows
  const SurpOff so = surprise_offsets(g);
  return so.per_unit % 4 == 0 && so.rp % 4 == 0 && so.g2 % 4 == 0 && so.maxcols % 4 == 0;
}

cudaError_t surprise_tc_readout(const Geom& g, const Chunk& ch, const Work& w, int buf, float* y, cudaStream_t st) {
  const SurpOff so = surprise_offsets(g);
  cudaError_t e = cudaFuncSetAttribute(k_surp_tc_g2, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_G);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_surp_tc_z, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_Z);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_surp_tc_y, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_Y);
  if (e != cudaSuccess) return e;
  // per unit, the band products of each read-out (four 16-token groups),
  // then the read-outs over their column blocks
  k_surp_tc_g2<<<dim3(4, g.units), NT, SMEM_G, st>>>(g, ch, w, so, 0, w.Zpre);
  k_surp_tc_z<<<dim3(g.hidden / 64, g.units), NT, SMEM_Z, st>>>(g, ch, w, buf, so, w.Zpre);
  k_surp_tc_g2<<<dim3(4, g.units), NT, SMEM_G, st>>>(g, ch, w, so, 1, w.Zpre);
  k_surp_tc_y<<<dim3(g.d_v / 32, g.units), NT, SMEM_Y, st>>>(g, ch, w, buf, so, w.Zpre, y);
  return cudaGetLastError();
}

cudaError_t surprise_tc_state(const Geom& g, const Chunk& ch, const Work& w, int buf, cudaStream_t st) {
  const SurpOff so = surprise_offsets(g);
  cudaError_t e = cudaFuncSetAttribute(k_surp_tc_state, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_S);
  if (e != cudaSuccess) return e;
  int tiles = 0;
  for (int m = 0; m < g.nmat; ++m) tiles += ((g.rows[m] + 127) / 128) * ((g.cols[m] + 127) / 128);
  k_surp_tc_state<<<dim3(tiles, g.units), NT, SMEM_S, st>>>(g, ch, w, buf, so);
  return cudaGetLastError();
}

}  // namespace atlas
