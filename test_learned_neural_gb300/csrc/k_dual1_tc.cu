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
// Per chunk, on each CTA (12 warps; warp 0 issues the MMAs):
//  1. generate the slice's R (C x FS) and window X (Kw x FS) tiles;
//  2. tensor cores: [R W^ | R S^] (M = 64, N = 128) and X W^ (M = 128,
//     N = 64), each as hi hi' + hi lo' + lo hi' (fp32 in TMEM); meanwhile
//     the owned rows of R X^T from the raw rows in closed form, the previous
//     chunk's read-out, and the bulk copies of the next chunk's rows;
//  3. the slice's partials go to their owners in the cluster (distributed
//     shared memory): rows t of B_t RW + D_t RS (owner t / YR), rows i of
//     X W^ (owner i / XR);
//  4. owners sum the NC slices in rank order, form dy rows (broadcast to
//     every CTA) and M = Cw * (R X^T) rows;
//  5. tensor cores: (cs_e dY)^T X, then (cw_e dY)^T X, for the chunk-end
//     state;
//  6. S' = A_e S^ - .., W' = B_e W^ + D_e S^ - .. into the TMEM masters and
//     the operand copies;
// the owned rows' y_t = Yp_t - (M dY)_t follow in the next chunk's step 2.
// Two cluster barriers per chunk order the exchanges.  Every mbarrier wait
// is bounded; a wait that gives up sets the status word and the CTA keeps
// the loop's barrier schedule without issuing further MMAs.
#include <cuda_bf16.h>

#include "atlas_common.cuh"
#include "tc.cuh"

namespace atlas {
namespace {

constexpr int NT = 384;                 // 12 warps: three per TMEM sub-partition
constexpr int FSM = 96, KWM = 80;       // max features per CTA, max window rows (padded)
constexpr int YS = 68;                  // row stride (floats) of the 64-wide exchange rows
constexpr int RECF = 16640;             // floats of the receive buffer (all senders)
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
constexpr int ORAW = ODYF + KWM * YS * 4;                  // raw rows (64 bytes): 64 queries, then Kw keys
constexpr int OVEC = ORAW + (64 + KWM) * 64;               // per-chunk gate vectors, by parity
constexpr int VECF = 296;
constexpr int OOWN = OVEC + 2 * VECF * 4;                  // owned rows' Cw, gamma, v (bf16)
constexpr int OOWN_G = OOWN + OWN_CW * 4;
constexpr int OOWN_V = OOWN_G + OWN_ROWS * 4;
constexpr int OTAB = OOWN_V + OWN_ROWS * 128;              // monomial table of the slice
constexpr int SMEM_BYTES = OTAB + FSM * 4;
static_assert(SMEM_BYTES + 1024 <= 227 * 1024, "shared memory map exceeds a CTA's limit");
static_assert(OREC % 16 == 0 && ODYF % 16 == 0 && ORAW % 16 == 0 && OVEC % 16 == 0 && OOWN_V % 16 == 0,
              "16-byte alignment");

// a gate-vector buffer is the block's tail from cs_e on: cs_e [kws], cw_e
// [kws], B_t [cp], D_t [cp], (A_e, B_e, D_e, 0)

// TMEM columns
constexpr uint32_t T_G1 = 0;     // [RW | RS], M = 64 layout
constexpr uint32_t T_XW = 224;   // X W^, M = 128 layout
constexpr uint32_t T_D1 = 0, T_D2 = 96;        // state corrections (M = 64, transposed)
constexpr uint32_t T_W = 288, T_S = 384;       // fp32 masters W^T, S^T (M = 64, transposed)

struct P1 {
  int nc, fs, kwp, yr, xr, nchunks;
  int blockf;   // floats of one sender's block in the receive buffer
  int own_pf;   // the owned rows' Cw, gamma, v fit the prefetch buffers
  CoefLayout L; // coefficient blocks (kws = kwp)
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
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// one arrival on *bar that also expects `bytes` of bulk-copy transactions
__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
// bulk copy global -> this CTA's shared memory (16-byte aligned, a multiple
// of 16 bytes), completing on *bar
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

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

// Bounded wait for a bulk-copy phase (every thread); a timeout is recorded.
__device__ __forceinline__ bool wait_data(uint64_t* bar, uint32_t parity, bool ok, int* status) {
  const bool good = tc::mbar_wait(bar, parity, kWait);
  const bool bad = __syncthreads_or(!good);
  if (bad && threadIdx.x == 0) atomicExch(status, ATLAS_ERR_TIMEOUT);
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

// Bulk copies (one thread) of chunk n's raw query rows and window-key rows
// (bf16, window-cache rows first) and its gate vectors, completing on *bar.
__device__ void prefetch_chunk(const Geom& g, const GenericIO& io, const float* coef, const P1& pp, int u, int n,
                               uint16_t* raw, float* vec, uint64_t* bar) {
  const Chunk ch = dual1_chunk_at(g, n * g.C);
  const int dk = g.d_k, C = g.C, rowb = 2 * dk;
  const int l0 = ch.lo + g.n_prev;                               // first key row of the window
  const int ncache = g.n_prev > l0 ? g.n_prev - l0 : 0;          // of them from the window cache
  const uint32_t vbytes = (uint32_t)(2 * pp.L.kws + 2 * pp.L.cp + 4) * 4u;
  mbar_expect(bar, (uint32_t)((C + ch.nw) * rowb) + vbytes);
  bulk_g2s(raw, (const uint16_t*)io.q + ((size_t)u * g.T + ch.s) * dk, (uint32_t)(C * rowb), bar);
  if (ncache > 0)
    bulk_g2s(raw + 64 * dk, (const uint16_t*)io.win_k + ((size_t)u * (g.c - 1) + (g.c - 1 - g.n_prev + l0)) * dk,
             (uint32_t)(ncache * rowb), bar);
  bulk_g2s(raw + (64 + ncache) * dk, (const uint16_t*)io.k + ((size_t)u * g.T + (l0 + ncache - g.n_prev)) * dk,
           (uint32_t)((ch.nw - ncache) * rowb), bar);
  const float* cb = coef + ((size_t)u * pp.nchunks + n) * pp.L.floats(C);
  bulk_g2s(vec + (n & 1) * VECF, cb + pp.L.o_cs(C), vbytes, bar);
}

// What the owner of rows t in [rank YR, +YR) and window rows i in
// [rank XR, +XR) reads in chunk n: Cw_t rows and v_i rows by bulk copies
// on *bar (one thread), gamma_i by cp.async (the same thread; 1 where the
// call has no gamma).  Nothing when they do not fit (the owner then reads
// them directly).
__device__ void prefetch_owner(const Geom& g, const GenericIO& io, const float* coef, const P1& pp, int u, int n,
                               int rank, float* ocw, float* og, uint16_t* ov, uint64_t* bar) {
  if (!pp.own_pf) {
    mbar_expect(bar, 0);
    return;
  }
  const Chunk ch = dual1_chunk_at(g, n * g.C);
  const int t0 = rank * pp.yr, t1 = min(g.C, t0 + pp.yr);
  const int i0 = rank * pp.xr, i1 = min(ch.nw, i0 + pp.xr);
  const int rowb = 2 * g.d_v, l0 = ch.lo + g.n_prev + i0;
  const int nrow = i1 > i0 ? i1 - i0 : 0;
  const int ncache = nrow > 0 && g.n_prev > l0 ? min(nrow, g.n_prev - l0) : 0;
  const uint32_t cwb = t1 > t0 ? (uint32_t)((t1 - t0) * pp.L.kws) * 4u : 0u;
  mbar_expect(bar, cwb + (uint32_t)(nrow * rowb));
  const float* cb = coef + ((size_t)u * pp.nchunks + n) * pp.L.floats(g.C);
  if (cwb) bulk_g2s(ocw, cb + (size_t)t0 * pp.L.kws, cwb, bar);
  if (ncache > 0)
    bulk_g2s(ov, (const uint16_t*)io.win_v + ((size_t)u * (g.c - 1) + (g.c - 1 - g.n_prev + l0)) * g.d_v,
             (uint32_t)(ncache * rowb), bar);
  if (nrow > ncache)
    bulk_g2s(ov + ncache * g.d_v,
             (const uint16_t*)io.v + ((size_t)u * g.T + (l0 + ncache - g.n_prev)) * g.d_v,
             (uint32_t)((nrow - ncache) * rowb), bar);
  for (int r = 0; r < pp.xr; ++r) {
    const int i = i0 + r;
    const float* gp = i < ch.nw ? gamma_ptr(g, io, u, ch.lo + g.n_prev + i) : nullptr;
    if (gp) cp4(og + r, gp, true);
    else og[r] = 1.f;
  }
  cp_commit();
}

// Raw rows (64 query rows, then Kw key rows) -> transposed xT[a][r] (bf16),
// with a = d_k the constant 1 and a = d_k + 1 the constant 0.
constexpr int RT = 64 + KWM;
__device__ void transpose_raw(int dk, const uint16_t* raw, uint16_t* xT) {
  const int pieces = dk / 8;
  for (int e = threadIdx.x; e < RT * pieces; e += NT) {
    const int r = e / pieces, pc = e % pieces;
    const uint4 v = *reinterpret_cast<const uint4*>(raw + r * dk + pc * 8);
    const uint16_t* h = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
    for (int k = 0; k < 8; ++k) xT[(pc * 8 + k) * RT + r] = h[k];
  }
  for (int r = threadIdx.x; r < RT; r += NT) {
    xT[dk * RT + r] = 0x3F80;   // bf16 1.0
    xT[(dk + 1) * RT + r] = 0;
  }
}

// The slice's query rows (R, 64 x FS) and window rows (X, Kw x FS) of the
// monomial map, split bf16, from x' = [x, 1, 0]: feature f is s_f x'_a x'_b
// with (a, b, s_f = 1 or 1/2) from the slice's table.  A group of 32
// threads keeps one chunk of 8 features' table entries in registers and
// walks the rows (consecutive rows in consecutive lanes: the reads of xT and
// the 16-byte stores of a warp fall in distinct banks).
__device__ void generate_tiles(const Geom& g, const Chunk& ch, const P1& pp, int rgs, const uint16_t* xT,
                               const uint32_t* tab, uint8_t* r_hi, uint8_t* r_lo, uint8_t* x_hi, uint8_t* x_lo) {
  const int nch = pp.fs / 8, rows = 64 + pp.kwp, ngroups = NT / 32;
  const int lane = threadIdx.x % 32;
  for (int c = threadIdx.x / 32; c < nch; c += ngroups) {
    const int c8 = c * 8;
    const uint16_t* pa[8];
    const uint16_t* pb[8];
    float sc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t t = tab[c8 + k];
      pa[k] = xT + (t & 255u) * RT;
      pb[k] = xT + ((t >> 8) & 255u) * RT;
      sc[k] = (t >> 16) ? 0.5f : 1.f;
    }
#pragma unroll 2
    for (int r = lane; r < rows; r += 32) {
      const bool isq = r < 64;
      const int i = r - 64;
      const bool valid = isq ? r < g.C : i < ch.nw;
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float p = tc::bf2f(pa[k][r]) * tc::bf2f(pb[k][r]) * sc[k];
        v[k] = valid ? p : 0.f;
      }
      if (isq) put8(r_hi, r_lo, tc::core_offset(r, c8, rgs), v);
      else put8(x_hi, x_lo, tc::core_offset(i, c8, rgs), v);
    }
  }
}

// dY (fp32 rows) times a per-row scale -> a split MN-major operand tile;
// threads [first, first + count)
__device__ void scale_dy(const float* dyf, const float* sc, int kwp, uint8_t* hi, uint8_t* lo, int first, int count) {
  for (int e = (int)threadIdx.x - first; e < kwp * 8; e += count) {
    const int i = e % kwp, c8 = (e / kwp) * 8;
    const float4 v0 = *reinterpret_cast<const float4*>(dyf + i * YS + c8);
    const float4 v1 = *reinterpret_cast<const float4*>(dyf + i * YS + c8 + 4);
    const float a = sc[i];
    const float sa[8] = {a * v0.x, a * v0.y, a * v0.z, a * v0.w, a * v1.x, a * v1.y, a * v1.z, a * v1.w};
    put8(hi, lo, tc::core_offset(i, c8, 1024), sa);
  }
}

// R X^T on the owned rows t = rank YR + r, from the raw rows (xT):
// phi(q) . phi(k) = 1 + q.k + ((q.k)^2 + sum_a (q_a k_a)^2) / 8 for the
// degree-2 map [1, x_a, x_a x_b / 2 (a <= b)] (sum_{a<=b} z_a z_b =
// ((sum z)^2 + sum z^2) / 2 with z_a = q_a k_a), q.k for the identity map;
// zero outside the chunk's tokens and window rows.  Four window rows per
// thread; vt is the thread's index among the count taking part.
__device__ void rx_rows(const Geom& g, const P1& pp, int rank, const Chunk& ch, const uint16_t* xT, float* rx,
                        int vt, int count) {
  const int KWP = pp.kwp, nq = KWP / 4;
  for (int e = vt; e < pp.yr * nq; e += count) {
    const int r = e / nq, i0 = (e % nq) * 4, t = rank * pp.yr + r;
    if (t >= 64) break;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (t < g.C) {
      float dot[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int a = 0; a < g.d_k; ++a) {
        const float xq = tc::bf2f(xT[a * RT + t]);
        const uint2 kk = *reinterpret_cast<const uint2*>(xT + a * RT + 64 + i0);
        const float xk[4] = {__uint_as_float(kk.x << 16), __uint_as_float(kk.x & 0xFFFF0000u),
                             __uint_as_float(kk.y << 16), __uint_as_float(kk.y & 0xFFFF0000u)};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float z = xq * xk[k];
          dot[k] += z;
          sq[k] += z * z;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (i0 + k < ch.nw) v[k] = g.p == 2 ? 1.f + dot[k] + 0.125f * (dot[k] * dot[k] + sq[k]) : dot[k];
    }
    *reinterpret_cast<float4*>(rx + r * (KWP + 4) + i0) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// y of the owned rows t = rank YR + r of chunk ch: Yp_t - (M dY)_t from the
// owned sums (mine) and dY.  A thread takes four rows, four columns and
// half of the window rows (one dY load serves four rows; lanes l and l ^ 16
// hold the two halves).  Threads [first, first + count), count a multiple
// of 32.
__device__ void readout_rows(const Geom& g, const GenericIO& io, const P1& pp, int u, int rank, const Chunk& ch,
                             const float* mine, const float* dyf, int first, int count) {
  const int KWP = pp.kwp, oRX = pp.yr * YS, nb = (pp.yr + 3) / 4, half = KWP / 2;
  for (int e = (int)threadIdx.x - first; e < nb * 32; e += count) {   // whole warps per iteration
    const int rb = e >> 5, h = (e >> 4) & 1, j0 = (e & 15) * 4;
    float4 acc[4];
    const float* m[4];
    bool live[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = rb * 4 + q;
      live[q] = r < pp.yr && rank * pp.yr + r < g.C && j0 < g.d_v;
      acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      m[q] = mine + oRX + (live[q] ? r : 0) * (KWP + 4);
    }
#pragma unroll 4
    for (int i = h * half; i < (h + 1) * half; ++i) {
      const float4 d = *reinterpret_cast<const float4*>(dyf + i * YS + j0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float mi = m[q][i];
        acc[q].x += mi * d.x;
        acc[q].y += mi * d.y;
        acc[q].z += mi * d.z;
        acc[q].w += mi * d.w;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[q].x += __shfl_xor_sync(0xffffffffu, acc[q].x, 16);
      acc[q].y += __shfl_xor_sync(0xffffffffu, acc[q].y, 16);
      acc[q].z += __shfl_xor_sync(0xffffffffu, acc[q].z, 16);
      acc[q].w += __shfl_xor_sync(0xffffffffu, acc[q].w, 16);
    }
    if (h == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (live[q]) {
          const int r = rb * 4 + q;
          const float4 yp = *reinterpret_cast<const float4*>(mine + r * YS + j0);
          *reinterpret_cast<float4*>(io.y + ((size_t)u * g.T + ch.s + rank * pp.yr + r) * g.d_v + j0) =
              make_float4(yp.x - acc[q].x, yp.y - acc[q].y, yp.z - acc[q].z, yp.w - acc[q].w);
        }
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(NT, 1) k_dual1_tc(Geom g, Work w, GenericIO io, const float* coef, P1 pp,
                                                     int fbuf) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar, bar_ch, bar_own;   // MMA groups, chunk rows, owner data
  __shared__ uint32_t tbase_s;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int q4 = warp & 3, hw = warp >> 2;        // TMEM sub-partition, column group (0-2)
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
  // R X^T of the chunk: in another sender's R X^T region (no sender writes
  // those), so the previous chunk's M stays readable meanwhile
  float* rxb = rec + ((rank + 1) % NC) * pp.blockf + oRX;
  const int vCS = 0, vCW = pp.L.kws, vBT = 2 * pp.L.kws, vDT = vBT + pp.L.cp, vABD = vDT + pp.L.cp;

  if (warp == 0) tc::tmem_alloc(&tbase_s, 512);
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init(&bar_ch, 1);
    tc::mbar_init(&bar_own, 1);
  }
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
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = tbase_s;

  // the call's initial W, S slice -> fp32 masters (transposed) and operand copies
  {
    const float* Wg = w.Wst[0][0] + (size_t)u * g.F * dv;
    const float* Sg = w.Sst[0][0] + (size_t)u * g.F * dv;
    const int j = 16 * q4 + (lane & 15);
    for (int cb = 32 * hw; cb < FS; cb += 96) {
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
  // bulk copies: chunk(0) here; chunk(n + 1) and owner(n) while chunk n's
  // first MMA group runs (thread 128), both complete before barrier B1 of
  // chunk n
  if (tid == 128) prefetch_chunk(g, io, coef, pp, u, 0, raw, vec, &bar_ch);
  tc::fence_before_sync();
  cluster_barrier();   // every CTA of the cluster runs: its shared memory takes peer stores from here on
  tc::fence_after_sync();

  bool ok = true;
  uint32_t phase = 0;
  for (int n = 0; n < pp.nchunks; ++n) {
    const Chunk ch = dual1_chunk_at(g, n * C);
    const float* vb = vec + (n & 1) * VECF;
    const bool more = n + 1 < pp.nchunks;
    ok = wait_data(&bar_ch, n & 1, ok, w.status);   // chunk(n)'s rows and gate vectors
    uint16_t* xT = reinterpret_cast<uint16_t*>(d_hi);   // the dY tiles are free until step 5
    transpose_raw(dk, raw, xT);
    __syncthreads();
    generate_tiles(g, ch, pp, rgs, xT, tab, r_hi, r_lo, x_hi, x_lo);

    // 2. partial products of the slice; meanwhile the next chunk's rows and
    //    this chunk's owner data load, and the previous chunk's owned rows
    //    are read out
    sync_mma();
    if (warp == 0) {   // the MMA warp does nothing else meanwhile
      if (lane == 0 && ok) {
        mma_split(tb + T_G1, kmajor(r_hi, r_lo, rgs), kmajor(b_hi, b_lo, rgs),
                  tc::idesc_f16(64, 128, 1, 0, 0), FS);
        mma_split(tb + T_XW, kmajor(x_hi, x_lo, rgs), kmajor(b_hi, b_lo, rgs), tc::idesc_f16(128, 64, 1, 0, 0), FS);
        tc::mma_commit(&bar);
      }
      __syncwarp();
    } else {
      if (tid == 128) {
        if (more) prefetch_chunk(g, io, coef, pp, u, n + 1, raw, vec, &bar_ch);
        prefetch_owner(g, io, coef, pp, u, n, (int)rank, ocw, og, ov, &bar_own);
      }
      // warps 1-3 read out chunk n - 1, warps 5-11 form R X^T of chunk n
      // (warp 4 issues the copies).  One CTA: R X^T goes where the read-out
      // reads M, after it.
      const int vt = (warp - 5) * 32 + lane;
      if (NC > 1) {
        if (warp < 4) {
          if (n > 0) readout_rows(g, io, pp, u, (int)rank, dual1_chunk_at(g, (n - 1) * C), mine, dyf, 32, 96);
        } else if (warp > 4) {
          rx_rows(g, pp, (int)rank, ch, xT, rxb, vt, NT - 160);
        }
      } else {
        if (n > 0) readout_rows(g, io, pp, u, (int)rank, dual1_chunk_at(g, (n - 1) * C), mine, dyf, 32, NT - 32);
        asm volatile("bar.sync 1, %0;" ::"r"(NT - 32) : "memory");
        rx_rows(g, pp, (int)rank, ch, xT, rxb, tid - 32, NT - 32);
      }
    }
    ok = wait_group(&bar, phase, ok, w.status);

    // 3. partials to their owners: rows t of Yp = B_t RW + D_t RS and of R X^T
    //    (owner t / YR), rows i of X W^ (owner i / XR)
    {
      const uint32_t blk = tc::smem_u32(rec) + rank * (uint32_t)pp.blockf * 4u;   // this sender's block
      const int t = 16 * q4 + (lane & 15), owner = t / YR, tr = t % YR;
      if (hw < 2) {   // Yp columns [32 hw, 32 hw + 32)
        const float bt = t < C ? vb[vBT + t] : 0.f, dt = t < C ? vb[vDT + t] : 0.f;
        const int cb = 32 * hw;
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
      } else if (32 * q4 < KWP) {   // X W^ rows in the M = 128 lanes: i = 32 q4 + lane
        for (int cb = 0; cb < 64; cb += 32) {
          float a[32];
          tc::tmem_ld16(tb + lane_base + T_XW + cb, a);
          tc::tmem_ld16(tb + lane_base + T_XW + cb + 16, a + 16);
          tc::tmem_ld_wait();
          const int i = 32 * q4 + lane;
          if (i < KWP) {
            const uint32_t dst = peer_addr(blk + (uint32_t)(oXW + (i % XR) * YS + cb) * 4u, i / XR);
#pragma unroll
            for (int k = 0; k < 32; k += 4) st_peer4(dst + 4u * k, a[k], a[k + 1], a[k + 2], a[k + 3]);
          }
        }
      }
    }
    cp_wait<0>();   // owner(n)'s gamma (thread 128)
    ok = wait_data(&bar_own, n & 1, ok, w.status);   // owner(n)'s Cw and v rows
    tc::fence_before_sync();
    cluster_barrier();   // B1: every partial has arrived
    tc::fence_after_sync();

    // 4. the owned rows: sums over the NC senders in rank order, four
    //    columns per thread
    {
      const float* Cwg = coef + ((size_t)u * pp.nchunks + n) * pp.L.floats(C);
      for (int e = tid; e < YR * 16; e += NT) {
        const int r = e >> 4, j0 = (e & 15) * 4;
        if ((int)rank * YR + r >= 64) break;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int src = 0; src < NC; ++src) {
          const float4 v = *reinterpret_cast<const float4*>(rec + src * pp.blockf + r * YS + j0);
          s.x += v.x;
          s.y += v.y;
          s.z += v.z;
          s.w += v.w;
        }
        *reinterpret_cast<float4*>(mine + r * YS + j0) = s;
      }
      for (int e = tid; e < YR * KWP; e += NT) {   // M = Cw * (R X^T), in place
        const int r = e / KWP, i = e % KWP, t = (int)rank * YR + r;
        if (t >= 64) break;
        float cw = 0.f;
        if (t < C && i < ch.nw) cw = pp.own_pf ? ocw[r * pp.L.kws + i] : Cwg[(size_t)t * pp.L.kws + i];
        mine[oRX + r * (KWP + 4) + i] = cw * rxb[r * (KWP + 4) + i];
      }
      for (int e = tid; e < XR * 16; e += NT) {
        const int r = e % XR, j0 = (e / XR) * 4, i = (int)rank * XR + r;
        if (i >= KWP) continue;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (i < ch.nw) {
          float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int src = 0; src < NC; ++src) {
            const float4 v = *reinterpret_cast<const float4*>(rec + src * pp.blockf + oXW + r * YS + j0);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
          }
          const int l = ch.lo + g.n_prev + i;
          float gm = 1.f;
          if (pp.own_pf) {
            gm = og[r];
          } else {
            const float* gp = gamma_ptr(g, io, u, l);
            if (gp) gm = *gp;
          }
          const uint16_t* vr = pp.own_pf ? ov + r * dv : v_row(g, io, u, l);
          const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (j0 + k < dv) d[k] = 2.f * gm * (sv[k] - tc::bf2f(vr[j0 + k]));
        }
        const uint32_t loc = tc::smem_u32(dyf + i * YS + j0);
        for (int p = 0; p < NC; ++p) st_peer4(peer_addr(loc, p), d[0], d[1], d[2], d[3]);
      }
    }
    tc::fence_before_sync();
    cluster_barrier();   // B2: every dy row has arrived
    tc::fence_after_sync();

    // 5. chunk-end corrections on the tensor cores: (cs_e dY)^T X and
    //    (cw_e dY)^T X, the second operand in the R tile (free since the
    //    first group completed)
    scale_dy(dyf, vb + vCS, KWP, d_hi, d_lo, 0, NT);
    sync_mma();
    const uint32_t ids = tc::idesc_f16(64, FS, 1, 1, 1);
    if (warp == 0) {   // (cs_e dY)^T X while the other warps scale for the second product
      if (lane == 0 && ok) mma_split(tb + T_D1, mnmajor(d_hi, d_lo, 1024), mnmajor(x_hi, x_lo, rgs), ids, KWP);
      __syncwarp();
    } else {
      scale_dy(dyf, vb + vCW, KWP, r_hi, r_hi + DYT, 32, NT - 32);
    }
    sync_mma();
    if (tid == 0 && ok) {
      mma_split(tb + T_D2, mnmajor(r_hi, r_hi + DYT, 1024), mnmajor(x_hi, x_lo, rgs), ids, KWP);
      tc::mma_commit(&bar);   // covers both products
    }
    ok = wait_group(&bar, phase, ok, w.status);

    // 6. chunk-end state of the slice
    {
      const float Ae = vb[vABD], Be = vb[vABD + 1], De = vb[vABD + 2];
      const int j = 16 * q4 + (lane & 15);
      for (int cb = 32 * hw; cb < FS; cb += 96) {
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

  // the last chunk's owned rows, then the call's final W, S slice
  readout_rows(g, io, pp, u, (int)rank, dual1_chunk_at(g, (pp.nchunks - 1) * C), mine, dyf, 0, NT);
  {
    float* Wg = w.Wst[fbuf][0] + (size_t)u * g.F * dv;
    float* Sg = w.Sst[fbuf][0] + (size_t)u * g.F * dv;
    const int j = 16 * q4 + (lane & 15);
    for (int cb = 32 * hw; cb < FS; cb += 96) {
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
  p.L = coef_layout_tc(g);
  p.own_pf = p.yr * p.L.kws <= OWN_CW && p.xr <= OWN_ROWS;
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
  // 16-byte copies of the raw key, query and value rows; 16-byte stores of y
  return ((uintptr_t)io.q % 16 == 0) && ((uintptr_t)io.k % 16 == 0) && ((uintptr_t)io.v % 16 == 0) &&
         ((uintptr_t)io.win_k % 16 == 0) && ((uintptr_t)io.win_v % 16 == 0) && ((uintptr_t)io.y % 16 == 0);
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
