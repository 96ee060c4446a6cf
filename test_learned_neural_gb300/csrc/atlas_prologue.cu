// The stage in front of the memory: projection (one GEMM of our own into the
// workspace: TMA-fed tcgen05 tiles for bf16 inputs, k_proj_gemm.cu), then
// one kernel for the causal depthwise convolution, the q/k normalisation,
// the gate heads, the layout change to [B][H][T][d] and the outgoing
// convolution cache.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <string>

#include "../../include/atlas_prologue.h"

namespace {

constexpr int kTok = 64;        // tokens per CTA
constexpr int kThreads = 256;
constexpr int kMaxTaps = 8;
constexpr int kMaxHeadCh = 512; // 2 d_k + d_v

struct PGeom {
  int D, H, dk, dv, K, G, Ch, Nc, N, dtype;
  float theta_max;
  int Np;     // row stride of the fp32 projection: N rounded up to 4 floats (16 bytes)
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}

size_t pro_smem_bytes(const PGeom& p) {
  // U rows with the K-1 halo, then the taps [K][Ch]
  return ((size_t)(kTok + p.K - 1) * p.Ch + (size_t)p.K * p.Ch) * sizeof(float);
}

// global channel of the head's local channel c (q: [0, dk), k: [dk, 2dk), v: [2dk, Ch))
__device__ __forceinline__ int head_channel(const PGeom& p, int h, int c) {
  if (c < p.dk) return h * p.dk + c;
  if (c < 2 * p.dk) return p.H * p.dk + h * p.dk + (c - p.dk);
  return 2 * p.H * p.dk + h * p.dv + (c - 2 * p.dk);
}

__device__ __forceinline__ void store_out(void* base, size_t i, float v, int dtype) {
  if (dtype == ATLAS_BF16)
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(base)[i] = v;
}

// P consecutive floats from shared memory (P = 1 or 2; 2: 8-byte aligned)
template <int P>
__device__ __forceinline__ void lds(float* out, const float* src) {
  if constexpr (P == 2) {
    const float2 f = *reinterpret_cast<const float2*>(src);
    out[0] = f.x;
    out[1] = f.y;
  } else {
    out[0] = *src;
  }
}

// P consecutive outputs at element i (P = 2: i even, base aligned to 2 elements)
template <int P>
__device__ __forceinline__ void store_vec(void* base, size_t i, const float* v, int dtype) {
  if constexpr (P == 2) {
    if (dtype == ATLAS_BF16)
      *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(base) + i) = __floats2bfloat162_rn(v[0], v[1]);
    else
      *reinterpret_cast<float2*>(reinterpret_cast<float*>(base) + i) = make_float2(v[0], v[1]);
  } else {
    store_out(base, i, v[0], dtype);
  }
}

// One CTA per (64-token tile, head, batch row).  The head's projected rows
// (with the K-1 halo) come into shared memory by cp.async, 16-byte copies
// where every segment is a multiple of 4 floats (vec), all in flight before
// one wait.  Then lane l of every warp owns the head's channels P l + 32 P i
// (+0 .. P-1; P = 2 where the head widths are even: paired loads and
// stores); warp w takes the 8 consecutive token rows [8w, 8w + 8) in groups
// of RG, sliding a register window of RG + K - 1 rows down each channel, so
// the q and k norms are warp reductions and no row leaves registers between
// the convolution and the store.  KT = K at compile time (the pages' 4), or
// 0 for any K <= 8.
template <int kSlots, int KT, int P>
__global__ void __launch_bounds__(kThreads, kSlots * P <= 6 ? 4 : 1) k_prologue(PGeom p, int T, const float* __restrict__ U,
                                                       const float* __restrict__ conv_w,
                                                       const float* __restrict__ gate_b,
                                                       const float* __restrict__ cache, void* q, void* k, void* v,
                                                       float* theta, float* eta, float* alpha, float* gamma,
                                                       float* cache_out, int vec) {
  extern __shared__ float sm[];
  const int t0 = blockIdx.x * kTok, h = blockIdx.y, b = blockIdx.z;
  const int K = KT > 0 ? KT : p.K, Ch = p.Ch, rows = kTok + K - 1;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  constexpr int NW = kThreads / 32;
  float* Us = sm;                          // [rows][Ch]: token t0 - (K-1) + r
  float* taps = Us + (size_t)rows * Ch;    // [K][Ch]: tap s weighs token t - (K-1) + s
  const size_t urow = (size_t)b * T;       // first U row of this batch row
  int gcs[kSlots];                         // global channel of each owned slot's first channel
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    const int c = P * lane + 32 * P * i;
    gcs[i] = c < Ch ? head_channel(p, h, c) : 0;
  }
  for (int j = warp; j < K; j += NW)
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int c = P * lane + 32 * P * i;
      if (c < Ch)
#pragma unroll
        for (int e = 0; e < P; ++e) taps[j * Ch + c + e] = conv_w[(size_t)(gcs[i] + e) * K + j];
    }
  {
    const int wv = vec ? 4 : 1, nv = Ch / wv;
    for (int r = warp; r < rows; r += NW) {
      const int t = t0 - (K - 1) + r;
      const float* srow = nullptr;
      if (t >= 0 && t < T)
        srow = U + (urow + t) * p.Np;
      else if (t < 0 && cache)
        srow = cache + ((size_t)b * (K - 1) + (K - 1) + t) * p.Nc;
      for (int cc = lane; cc < nv; cc += 32) {
        const int c = cc * wv;
        float* dst = Us + r * Ch + c;
        if (srow) {
          if (vec)
            cp_async16(dst, srow + head_channel(p, h, c));
          else
            cp_async4(dst, srow + head_channel(p, h, c));
        } else {
          for (int q4 = 0; q4 < wv; ++q4) dst[q4] = 0.f;
        }
      }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  const size_t uh = (size_t)b * p.H + h;   // (batch, head) index of the outputs
  constexpr int RPW = kTok / NW;           // rows per warp
  constexpr int RG = kSlots * P <= 8 ? 4 : 2;   // rows per register group
  for (int g0 = warp * RPW; g0 < warp * RPW + RPW; g0 += RG) {
    if (t0 + g0 >= T) break;
    float val[RG][kSlots][P];
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int c = P * lane + 32 * P * i;
      if (c < Ch) {
        float tp[kMaxTaps][P], win[RG + kMaxTaps - 1][P];
#pragma unroll
        for (int s2 = 0; s2 < kMaxTaps; ++s2) {
          if (s2 < K) {
            lds<P>(tp[s2], taps + s2 * Ch + c);
          } else {
#pragma unroll
            for (int e = 0; e < P; ++e) tp[s2][e] = 0.f;
          }
        }
#pragma unroll
        for (int m = 0; m < RG + kMaxTaps - 1; ++m) {
          if (m < RG + K - 1) {
            lds<P>(win[m], Us + (g0 + m) * Ch + c);
          } else {
#pragma unroll
            for (int e = 0; e < P; ++e) win[m][e] = 0.f;
          }
        }
#pragma unroll
        for (int rr = 0; rr < RG; ++rr)
#pragma unroll
          for (int e = 0; e < P; ++e) {
            float acc = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < kMaxTaps; ++s2)
              if (s2 < K) acc += tp[s2][e] * win[rr + s2][e];
            val[rr][i][e] = acc;
          }
      } else {
#pragma unroll
        for (int rr = 0; rr < RG; ++rr)
#pragma unroll
          for (int e = 0; e < P; ++e) val[rr][i][e] = 0.f;
      }
    }
#pragma unroll
    for (int rr = 0; rr < RG; ++rr) {
      const int t = t0 + g0 + rr;   // warp-uniform
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        const int c = P * lane + 32 * P * i;   // a slot never straddles q, k, v (even widths when P = 2)
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < P; ++e) ss += val[rr][i][e] * val[rr][i][e];
        if (c < p.dk) sq += ss;
        else if (c < 2 * p.dk) sk += ss;
      }
      for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      if (t >= T) continue;
      const float iq = 1.f / fmaxf(sqrtf(sq), 1e-12f), ik = 1.f / fmaxf(sqrtf(sk), 1e-12f);
      const size_t rk = (uh * T + t) * p.dk, rv = (uh * T + t) * p.dv;
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        const int c = P * lane + 32 * P * i;
        if (c >= Ch) continue;
        float o[P];
        if (c < p.dk) {
#pragma unroll
          for (int e = 0; e < P; ++e) o[e] = val[rr][i][e] * iq;
          store_vec<P>(q, rk + c, o, p.dtype);
        } else if (c < 2 * p.dk) {
#pragma unroll
          for (int e = 0; e < P; ++e) o[e] = val[rr][i][e] * ik;
          store_vec<P>(k, rk + (c - p.dk), o, p.dtype);
        } else {
          store_vec<P>(v, rv + (c - 2 * p.dk), val[rr][i], p.dtype);
        }
      }
    }
  }
  for (int e = threadIdx.x; e < p.G * kTok; e += kThreads) {
    const int g = e / kTok, r = e % kTok, t = t0 + r;
    if (t >= T) continue;
    const float l = U[(urow + t) * p.Np + p.Nc + (size_t)g * p.H + h] + gate_b[g * p.H + h];
    const float s = 1.f / (1.f + expf(-l));
    float* dst = g == 0 ? theta : g == 1 ? eta : g == 2 ? alpha : gamma;
    dst[uh * T + t] = g == 0 ? p.theta_max * s : s;
  }
  // the last K-1 projected rows (from the earlier cache where T < K-1), by
  // the CTA that holds token T-1
  if (cache_out && t0 <= T - 1 && T - 1 < t0 + kTok) {
    for (int i = warp; i < K - 1; i += NW) {
      const int t = T - (K - 1) + i;
      const float* src = nullptr;
      if (t >= 0)
        src = U + (urow + t) * p.Np;
      else if (cache)
        src = cache + ((size_t)b * (K - 1) + (K - 1) + t) * p.Nc;
      float* dst = cache_out + ((size_t)b * (K - 1) + i) * p.Nc;
#pragma unroll
      for (int s2 = 0; s2 < kSlots; ++s2)
        if (P * lane + 32 * P * s2 < Ch)
#pragma unroll
          for (int e = 0; e < P; ++e) dst[gcs[s2] + e] = src ? src[gcs[s2] + e] : 0.f;
    }
  }
}

}  // namespace

namespace atlas {
size_t proj_gemm_scratch(int N, int K, int bf16);
cudaError_t proj_gemm(const void* x, const void* W, int M, int N, int Np, int K, int bf16, float* U, void* wt,
                      int* status, cudaStream_t st, int* kind);
}

struct atlas_prologue_handle {
  atlas_prologue_config cfg;
  PGeom p;
  void* ws = nullptr;      // the fp32 projection, W_in transposed (tensor-core path), the status word
  size_t ws_bytes = 0;
  int* status = nullptr;
  cudaStream_t last_stream = nullptr;
  bool launched = false;
  int gemm_kind = -1;      // last projection: 1 tensor cores, 0 SIMT
  std::string err;
};

static thread_local std::string g_pro_create_err;

static int pfail(atlas_prologue_handle* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  return code;
}

extern "C" int atlas_prologue_create(const atlas_prologue_config* cfg, atlas_prologue_handle** out) {
  if (!out || !cfg) {
    g_pro_create_err = "cfg and out must be non-NULL";
    if (out) *out = nullptr;
    return ATLAS_ERR_INVALID_ARG;
  }
  *out = nullptr;
  const atlas_prologue_config& c = *cfg;
  auto bad = [&](int code, const char* why) {
    g_pro_create_err = why;
    return code;
  };
  if (c.D < 1 || c.H < 1 || c.d_k < 1 || c.d_v < 1) return bad(ATLAS_ERR_INVALID_ARG, "D, H, d_k, d_v must be >= 1");
  if (c.conv < 1) return bad(ATLAS_ERR_INVALID_ARG, "conv (taps) must be >= 1");
  if (c.with_gamma != 0 && c.with_gamma != 1) return bad(ATLAS_ERR_INVALID_ARG, "with_gamma must be 0 or 1");
  if (!(c.theta_max > 0.f) || !isfinite(c.theta_max)) return bad(ATLAS_ERR_INVALID_ARG, "theta_max must be > 0");
  if (c.qkv_dtype != ATLAS_F32 && c.qkv_dtype != ATLAS_BF16)
    return bad(ATLAS_ERR_INVALID_ARG, "qkv_dtype must be ATLAS_F32 or ATLAS_BF16");
  if (c.conv > kMaxTaps) return bad(ATLAS_ERR_UNSUPPORTED, "more than 8 convolution taps are not supported");
  if (2LL * c.d_k + c.d_v > kMaxHeadCh) return bad(ATLAS_ERR_UNSUPPORTED, "2 d_k + d_v > 512 per head is not supported");
  const long long Nc = (long long)c.H * (2 * c.d_k + c.d_v), N = Nc + (3LL + c.with_gamma) * c.H;
  if (N > (1LL << 24) || c.D > (1 << 24)) return bad(ATLAS_ERR_UNSUPPORTED, "projection wider than 2^24 is not supported");
  auto* h = new atlas_prologue_handle();
  h->cfg = c;
  h->p = PGeom{c.D, c.H, c.d_k, c.d_v, c.conv, 3 + c.with_gamma, 2 * c.d_k + c.d_v, (int)Nc, (int)N, c.qkv_dtype,
               c.theta_max, (int)((N + 3) / 4 * 4)};
  *out = h;
  return ATLAS_OK;
}

// bytes of the fp32 projection [B T][Np], rounded to 256
static size_t proj_bytes(const PGeom& p, int B, int T) { return ((size_t)B * T * p.Np * sizeof(float) + 255) / 256 * 256; }

extern "C" size_t atlas_prologue_workspace_bytes(const atlas_prologue_handle* h, int B, int T) {
  if (!h || B < 1 || T < 1) return 0;
  // the projection, W_in transposed for the tensor-core GEMM, the status word
  return proj_bytes(h->p, B, T) + atlas::proj_gemm_scratch(h->p.N, h->p.D, h->p.dtype == ATLAS_BF16) + 256;
}

extern "C" const char* atlas_prologue_last_error(const atlas_prologue_handle* h) {
  return h ? h->err.c_str() : g_pro_create_err.c_str();
}

extern "C" void atlas_prologue_destroy(atlas_prologue_handle* h) {
  if (!h) return;
  if (h->ws) cudaFree(h->ws);
  delete h;
}

extern "C" int atlas_prologue_forward(atlas_prologue_handle* h, const atlas_prologue_io* io, void* stream) {
  if (!h) return ATLAS_ERR_INVALID_ARG;
  if (!io) return pfail(h, ATLAS_ERR_INVALID_ARG, "io must be non-NULL");
  const PGeom& p = h->p;
  if (io->B < 1 || io->T < 1) return pfail(h, ATLAS_ERR_INVALID_ARG, "B and T must be >= 1");
  if (io->B > 65535) return pfail(h, ATLAS_ERR_UNSUPPORTED, "B > 65535 is not supported");
  if (!io->x || !io->W_in || !io->conv_w || !io->gate_b || !io->q || !io->k || !io->v || !io->theta || !io->eta ||
      !io->alpha)
    return pfail(h, ATLAS_ERR_INVALID_ARG, "x, W_in, conv_w, gate_b, q, k, v, theta, eta, alpha must be non-NULL");
  if ((p.G == 4) != (io->gamma != nullptr))
    return pfail(h, ATLAS_ERR_INVALID_ARG, "gamma must be given exactly when with_gamma is set");
  if (io->cache_out && io->cache_out == io->cache)
    return pfail(h, ATLAS_ERR_INVALID_ARG, "cache_out must not alias cache");
  const long long M = (long long)io->B * io->T;
  if (M > (1LL << 31) / 2 || M * p.N > (1LL << 40))
    return pfail(h, ATLAS_ERR_UNSUPPORTED, "B * T too large for one projection");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t need = atlas_prologue_workspace_bytes(h, io->B, io->T);
  if (h->ws_bytes < need) {
    if (h->ws) {
      cudaError_t e = cudaStreamSynchronize(st);
      if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
      cudaFree(h->ws);
      h->ws = nullptr;
      h->ws_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&h->ws, need);
    if (e != cudaSuccess) {
      cudaGetLastError();
      h->ws = nullptr;
      return pfail(h, ATLAS_ERR_OOM, "cudaMalloc(%zu) failed: %s", need, cudaGetErrorString(e));
    }
    h->ws_bytes = need;
    h->status = reinterpret_cast<int*>(reinterpret_cast<char*>(h->ws) + (need - 256));
    e = cudaMemsetAsync(h->status, 0, sizeof(int), st);
    if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  }
  // U [M][Np] = x [M][D] W_in [D][N], fp32 accumulation
  {
    const size_t wt_bytes = atlas::proj_gemm_scratch(p.N, p.D, p.dtype == ATLAS_BF16);
    void* wt = wt_bytes ? reinterpret_cast<char*>(h->ws) + proj_bytes(p, io->B, io->T) : nullptr;
    cudaError_t e = atlas::proj_gemm(io->x, io->W_in, (int)M, p.N, p.Np, p.D, p.dtype == ATLAS_BF16, (float*)h->ws,
                                     wt, h->status, st, &h->gemm_kind);
    if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "projection GEMM launch: %s", cudaGetErrorString(e));
  }
  const size_t smem = pro_smem_bytes(p);
  // channel pairs where both head widths are even and q, k, v are aligned
  // for paired stores
  const size_t es = p.dtype == ATLAS_BF16 ? 2 : 4;
  const bool pairs = p.dk % 2 == 0 && p.dv % 2 == 0 && (uintptr_t)io->q % (2 * es) == 0 &&
                     (uintptr_t)io->k % (2 * es) == 0 && (uintptr_t)io->v % (2 * es) == 0;
  decltype(&k_prologue<2, 4, 2>) kern;
  if (pairs) {
    const int slots = (p.Ch + 63) / 64;
    auto pick = [&](auto four, auto any) { return p.K == 4 ? four : any; };
    kern = slots <= 2   ? pick(k_prologue<2, 4, 2>, k_prologue<2, 0, 2>)
           : slots <= 3 ? pick(k_prologue<3, 4, 2>, k_prologue<3, 0, 2>)
           : slots <= 4 ? pick(k_prologue<4, 4, 2>, k_prologue<4, 0, 2>)
                        : pick(k_prologue<8, 4, 2>, k_prologue<8, 0, 2>);
  } else {
    const int slots = (p.Ch + 31) / 32;
    kern = slots <= 2 ? k_prologue<2, 0, 1> : slots <= 4 ? k_prologue<4, 0, 1>
         : slots <= 8 ? k_prologue<8, 0, 1> : k_prologue<16, 0, 1>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  dim3 grid((io->T + kTok - 1) / kTok, p.H, io->B);
  // 16-byte copies need every head segment, the projection's row stride and
  // the caller's cache rows on 16-byte boundaries
  const float* cache = p.K > 1 ? io->cache : nullptr;
  const int vec = p.dk % 4 == 0 && p.dv % 4 == 0 && ((uintptr_t)cache % 16) == 0;
  kern<<<grid, kThreads, smem, st>>>(p, io->T, (const float*)h->ws, io->conv_w, io->gate_b, cache, io->q, io->k,
                                     io->v, io->theta, io->eta, io->alpha, io->gamma,
                                     p.K > 1 ? io->cache_out : nullptr, vec);
  e = cudaGetLastError();
  if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "k_prologue launch: %s", cudaGetErrorString(e));
  h->last_stream = st;
  h->launched = true;
  return ATLAS_OK;
}

extern "C" int atlas_prologue_status(atlas_prologue_handle* h) {
  if (!h) return ATLAS_ERR_INVALID_ARG;
  if (!h->launched || !h->status) return ATLAS_OK;
  cudaError_t e = cudaStreamSynchronize(h->last_stream);
  if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  int s = 0;
  e = cudaMemcpy(&s, h->status, sizeof s, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return pfail(h, ATLAS_ERR_CUDA, "cudaMemcpy: %s", cudaGetErrorString(e));
  if (s != 0) {
    cudaMemset(h->status, 0, sizeof s);
    return pfail(h, ATLAS_ERR_TIMEOUT, "a device-side wait of the projection gave up (status %d)", s);
  }
  return ATLAS_OK;
}

extern "C" int atlas_prologue_last_gemm(const atlas_prologue_handle* h) { return h ? h->gemm_kind : -1; }
