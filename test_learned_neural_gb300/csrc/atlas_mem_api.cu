// Host side of the C ABI: config validation, workspace, launch sequence.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <string>

#include "atlas_common.cuh"


using namespace atlas;

struct atlas_mem_handle {
  atlas_mem_config cfg;
  Geom base;              // sizes that do not depend on the call
  void* ws = nullptr;     // device workspace
  size_t ws_bytes = 0;
  void* stage = nullptr;  // device staging for atlas_mem_forward_host
  size_t stage_bytes = 0;
  int* status = nullptr;  // device status word (inside ws)
  cudaStream_t last_stream = nullptr;
  bool launched = false;
  int launches = 0;       // kernel launches of the last forward
  std::string err;
  // Repeated identical calls of the multi-launch path replay a CUDA graph:
  // the second call with the same arguments (and workspace) captures the
  // launch sequence on a private stream, later ones launch the graph.
  cudaStream_t cap = nullptr;
  // host-buffer calls on the fused path: unit groups on their own streams,
  // so the copies of one group overlap the kernel of another
  static const int kGroups = 4;
  cudaStream_t pst[kGroups] = {};
  cudaEvent_t pev[2 * kGroups + 2] = {};
  cudaGraphExec_t gexec = nullptr;
  atlas_mem_io gkey{};    // arguments the graph was captured with
  void* gws = nullptr;
  int glaunches = 0;
  atlas_mem_io last_io{}; // arguments of the previous multi-launch call
  void* last_ws = nullptr;
  bool have_last = false;
};

// message of the last atlas_mem_create failure on this thread (no handle yet)
static thread_local std::string g_create_err;

static int fail(atlas_mem_handle* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  return code;
}

static constexpr size_t kSmemLimit = 227 * 1024;

static long long choose2(long long n) { return n * (n - 1) / 2; }

static int derive_geom(const atlas_mem_config& c, Geom* g, char* why, size_t why_n, bool* unsupported) {
  *unsupported = false;
  memset(g, 0, sizeof *g);
#define BAD(...)                            \
  do {                                      \
    snprintf(why, why_n, __VA_ARGS__);      \
    return 0;                               \
  } while (0)
  if (c.depth != 1 && c.depth != 2) BAD("depth must be 1 or 2 (got %d)", c.depth);
  if (c.d_k < 1 || c.d_v < 1) BAD("d_k and d_v must be >= 1");
  if (c.depth == 2 && c.hidden < 1) BAD("depth 2 needs hidden >= 1");
  if (c.C < 1) BAD("chunk size C must be >= 1");
  if (c.c < 1) BAD("Omega window c must be >= 1");
  if (c.p != 1 && c.p != 2) BAD("polynomial degree p must be 1 or 2 (got %d)", c.p);
  if (c.proj_dim < 0) BAD("proj_dim must be >= 0");
  if (c.ns_iters < 0) BAD("ns_iters must be >= 0");
  if (c.qkv_dtype != ATLAS_F32 && c.qkv_dtype != ATLAS_BF16) BAD("qkv_dtype must be ATLAS_F32 or ATLAS_BF16");
  if (c.readout != ATLAS_READOUT_POST && c.readout != ATLAS_READOUT_PRE)
    BAD("readout must be ATLAS_READOUT_POST or ATLAS_READOUT_PRE");
  if (c.ns_target != ATLAS_NS_MOMENTUM && c.ns_target != ATLAS_NS_SURPRISE)
    BAD("ns_target must be ATLAS_NS_MOMENTUM or ATLAS_NS_SURPRISE");
  if (c.ns_target == ATLAS_NS_SURPRISE && c.ns_iters > 0 && c.c > 32)
    BAD("Newton-Schulz on the surprise needs c <= 32 (its c x c core)");
  if (c.update != ATLAS_UPDATE_PER_TOKEN && c.update != ATLAS_UPDATE_CHUNKWISE)
    BAD("update must be ATLAS_UPDATE_PER_TOKEN or ATLAS_UPDATE_CHUNKWISE");
  if (c.update == ATLAS_UPDATE_CHUNKWISE && c.c != 1) BAD("the chunk-wise update has no Omega window: c must be 1");
  if (c.update == ATLAS_UPDATE_CHUNKWISE && c.ns_iters > 0 && c.ns_target != ATLAS_NS_MOMENTUM)
    BAD("the chunk-wise update orthogonalises the momentum only");
  long long poly = c.p == 1 ? c.d_k : 1 + c.d_k + choose2(c.d_k + 1);
  long long F = c.proj_dim ? c.proj_dim : poly;
  if (c.depth == 2 && F != c.d_v) BAD("depth 2 (residual memory) needs feature width %lld == d_v %d", F, c.d_v);
  g->depth = c.depth; g->d_k = c.d_k; g->d_v = c.d_v; g->hidden = c.depth == 2 ? c.hidden : 0;
  g->C = c.C; g->c = c.c; g->p = c.p; g->proj_dim = c.proj_dim; g->ns_iters = c.ns_iters;
  g->qkv_dtype = c.qkv_dtype;
  g->readout = c.readout;
  g->ns_target = c.ns_target;
  g->update = c.update;
  g->Kw = c.C + c.c - 1;
  if (c.depth == 1) {
    g->nmat = 1; g->rows[0] = (int)F; g->cols[0] = c.d_v;
  } else {
    g->nmat = 2; g->rows[0] = (int)F; g->cols[0] = c.hidden; g->rows[1] = c.hidden; g->cols[1] = c.d_v;
  }
  // limits of the kernels (valid configs beyond them are UNSUPPORTED)
  *unsupported = true;
  if (poly > 16384 || F > 8192 || c.d_v > 8192 || c.hidden > 8192) BAD("widths beyond 8192 features are not supported");
  if (g->Kw > 1024) BAD("C + c - 1 = %d > 1024 window rows per chunk is not supported", g->Kw);
  g->poly = (int)poly;
  g->F = (int)F;
  if (generic_smem_readout(*g) > kSmemLimit)
    BAD("memory widths too large for the on-chip working set");
  if ((size_t)(c.d_k + (c.proj_dim ? poly : 0)) * 4 > kSmemLimit) BAD("feature map too wide");
  if (c.ns_iters > 0 && c.ns_target == ATLAS_NS_MOMENTUM)
    for (int m = 0; m < g->nmat; ++m) {
      int rX = g->rows[m] < g->cols[m] ? g->rows[m] : g->cols[m];
      if (rX > 128) BAD("Newton-Schulz on matrices whose short side exceeds 128 is not supported");
    }
  *unsupported = false;
#undef BAD
  return 1;
}

// ------------------------------------------------------------ workspace map
struct Layout {
  size_t off[32];
  size_t total;
};

static size_t al(size_t x) { return (x + 255) & ~(size_t)255; }

// Sizes (in floats) of every workspace array, in Work order.
static Layout layout(const Geom& g, int units, int T) {
  Layout L{};
  const size_t U = units, Lr = (size_t)(g.c - 1) + T, Kw = g.Kw, h = g.hidden;
  size_t mat = 0;
  for (int m = 0; m < g.nmat; ++m) mat += (size_t)g.rows[m] * g.cols[m];
  size_t sizes[] = {
      U * Lr * g.F,                        // X
      U * Lr * g.d_v,                      // V
      U * Lr,                              // G
      U * (size_t)T * g.F,                 // R
      U * (size_t)g.rows[0] * g.cols[0],   // W buf0 m0
      U * (size_t)g.rows[1] * g.cols[1],   // W buf0 m1
      U * (size_t)g.rows[0] * g.cols[0],   // W buf1 m0
      U * (size_t)g.rows[1] * g.cols[1],   // W buf1 m1
      U * (size_t)g.rows[0] * g.cols[0],   // S buf0 m0
      U * (size_t)g.rows[1] * g.cols[1],   // S buf0 m1
      U * (size_t)g.rows[0] * g.cols[0],   // S buf1 m0
      U * (size_t)g.rows[1] * g.cols[1],   // S buf1 m1
      U * Kw * h,                          // Zpre
      U * Kw * h,                          // Aact
      U * Kw * h,                          // DZ
      U * Kw * g.d_v,                      // DY
      U * g.C * Kw,                        // Cs
      U * g.C * Kw,                        // Cw
      U * g.C, U * g.C, U * g.C,           // Ap Bp Dp
      g.ns_iters && g.ns_target == ATLAS_NS_MOMENTUM ? U * g.C * mat : 0,   // Ubuf
      U * (size_t)(g.c > 1 ? g.c - 1 : 0) * (g.d_k + g.d_v + 1),  // cache temp
      64,                                  // status
      g.depth == 2 ? U * ((size_t)(g.hidden + 63) / 64) * Kw * g.d_v  // tiled-gradient partial outputs
                   : dual1_split_floats(g, U, T),                       // depth 1: scaled dy + feature-slice partials
      g.ns_iters && g.ns_target == ATLAS_NS_SURPRISE ? surprise_floats(g, U) : 0,   // surprise NS scratch
      g.ns_iters && g.update == ATLAS_UPDATE_CHUNKWISE ? U * (size_t)T : 0,          // per-token decay (aeff)
      (features_tc_scratch_bytes(g) + 3) / 4,                                          // P transposed (bf16)
  };
  const int n = sizeof sizes / sizeof sizes[0];
  size_t o = 0;
  for (int i = 0; i < n; ++i) {
    L.off[i] = o;
    o += al(sizes[i] * sizeof(float));
  }
  L.total = o;
  return L;
}

static Work work_from(const Geom& g, void* base, const Layout& L, float** cache_tmp) {
  char* b = (char*)base;
  auto F = [&](int i) { return (float*)(b + L.off[i]); };
  Work w;
  w.X = F(0); w.V = F(1); w.G = F(2); w.R = F(3);
  w.Wst[0][0] = F(4); w.Wst[0][1] = F(5); w.Wst[1][0] = F(6); w.Wst[1][1] = F(7);
  w.Sst[0][0] = F(8); w.Sst[0][1] = F(9); w.Sst[1][0] = F(10); w.Sst[1][1] = F(11);
  w.Zpre = F(12); w.Aact = F(13); w.DZ = F(14); w.DY = F(15);
  w.Cs = F(16); w.Cw = F(17); w.Ap = F(18); w.Bp = F(19); w.Dp = F(20);
  w.Ubuf = F(21);
  *cache_tmp = F(22);
  w.status = (int*)F(23);
  w.gpart = F(24);
  w.surp = F(25);
  w.aeff = g.ns_iters && g.update == ATLAS_UPDATE_CHUNKWISE ? F(26) : nullptr;
  w.Pt = features_tc_scratch_bytes(g) ? (void*)F(27) : nullptr;
  return w;
}

// ------------------------------------------------------------------- API
extern "C" int atlas_mem_create(const atlas_mem_config* cfg, atlas_mem_handle** out) {
  if (!out || !cfg) {
    g_create_err = "cfg and out must be non-NULL";
    if (out) *out = nullptr;
    return ATLAS_ERR_INVALID_ARG;
  }
  *out = nullptr;
  Geom g;
  char why[256];
  bool unsup = false;
  if (!derive_geom(*cfg, &g, why, sizeof why, &unsup)) {
    g_create_err = why;
    return unsup ? ATLAS_ERR_UNSUPPORTED : ATLAS_ERR_INVALID_ARG;
  }
  atlas_mem_handle* h = new atlas_mem_handle();
  h->cfg = *cfg;
  h->base = g;
  *out = h;
  return ATLAS_OK;
}

extern "C" void atlas_mem_destroy(atlas_mem_handle* h) {
  if (!h) return;
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  if (h->cap) cudaStreamDestroy(h->cap);
  for (int i = 0; i < atlas_mem_handle::kGroups; ++i)
    if (h->pst[i]) cudaStreamDestroy(h->pst[i]);
  for (int i = 0; i < 2 * atlas_mem_handle::kGroups + 2; ++i)
    if (h->pev[i]) cudaEventDestroy(h->pev[i]);
  if (h->ws) cudaFree(h->ws);
  if (h->stage) cudaFree(h->stage);
  delete h;
}

extern "C" int atlas_mem_last_launches(const atlas_mem_handle* h) { return h ? h->launches : 0; }

extern "C" const char* atlas_mem_last_error(const atlas_mem_handle* h) {
  return h ? h->err.c_str() : g_create_err.c_str();
}

extern "C" size_t atlas_mem_workspace_bytes(const atlas_mem_handle* h, int B, int H, int T) {
  if (!h || B <= 0 || H <= 0 || T <= 0) return 0;
  return layout(h->base, B * H, T).total;
}

static int check_io(atlas_mem_handle* h, const atlas_mem_io* io) {
  if (!io) return fail(h, ATLAS_ERR_INVALID_ARG, "io is NULL");
  const Geom& g = h->base;
  if (io->B <= 0 || io->H <= 0 || io->T <= 0) return fail(h, ATLAS_ERR_INVALID_ARG, "B, H, T must be > 0");
  if ((long long)io->B * io->H > (1 << 20)) return fail(h, ATLAS_ERR_UNSUPPORTED, "more than 2^20 units");
  if (io->T % g.C != 0) return fail(h, ATLAS_ERR_UNSUPPORTED, "T = %d is not a multiple of C = %d", io->T, g.C);
  if (!io->q || !io->k || !io->v || !io->theta || !io->eta || !io->alpha || !io->y)
    return fail(h, ATLAS_ERR_INVALID_ARG, "q, k, v, theta, eta, alpha and y must be non-NULL");
  for (int m = 0; m < g.nmat; ++m)
    if (!io->W0[m] || !io->S0[m] || !io->W_out[m] || !io->S_out[m])
      return fail(h, ATLAS_ERR_INVALID_ARG, "W0/S0/W_out/S_out[%d] must be non-NULL", m);
  if (g.proj_dim && !io->P) return fail(h, ATLAS_ERR_INVALID_ARG, "proj_dim > 0 needs P");
  if (io->win_len < 0 || io->win_len > g.c - 1)
    return fail(h, ATLAS_ERR_INVALID_ARG, "win_len = %d outside [0, c-1 = %d]", io->win_len, g.c - 1);
  if (io->win_len > 0 && (!io->win_k || !io->win_v))
    return fail(h, ATLAS_ERR_INVALID_ARG, "win_len > 0 needs win_k and win_v");
  return ATLAS_OK;
}

#define CUDA_TRY(call)                                                                          \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess) return fail(h, ATLAS_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

static int ensure_workspace(atlas_mem_handle* h, size_t bytes) {
  if (h->ws_bytes >= bytes) return ATLAS_OK;
  const char* inj = getenv("ATLAS_INJECT_ALLOC_FAILURE");
  if (inj && inj[0] == '1') return fail(h, ATLAS_ERR_OOM, "workspace allocation of %zu bytes failed (injected)", bytes);
  if (h->ws) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(h, ATLAS_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_bytes = 0;
  }
  cudaError_t e = cudaMalloc(&h->ws, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return fail(h, ATLAS_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  e = cudaMemset(h->ws, 0, bytes);
  if (e != cudaSuccess) return fail(h, ATLAS_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
  h->ws_bytes = bytes;
  return ATLAS_OK;
}

// the multi-launch path: state in, per-chunk kernels, state and cache out
static int run_generic(atlas_mem_handle* h, const Geom& g, const Work& w, const atlas_mem_io* io, float* cache_tmp,
                       cudaStream_t st, int* nl_out) {
  int nl = 0;
  const bool ns_tc = ns_tc_supported(g);   // keeps S transposed for tall matrices
  for (int m = 0; m < g.nmat; ++m) {
    const size_t bytes = (size_t)g.units * g.rows[m] * g.cols[m] * sizeof(float);
    CUDA_TRY(cudaMemcpyAsync(w.Wst[0][m], io->W0[m], bytes, cudaMemcpyDeviceToDevice, st));
    if (ns_tc) CUDA_TRY(ns_tc_state_in(g, m, io->S0[m], w.Sst[0][m], st));
    else CUDA_TRY(cudaMemcpyAsync(w.Sst[0][m], io->S0[m], bytes, cudaMemcpyDeviceToDevice, st));
  }
  GenericIO gio{io->q, io->k, io->v, io->P, io->win_len ? io->win_k : nullptr, io->win_len ? io->win_v : nullptr,
                io->theta, io->eta, io->alpha, io->gamma, io->win_len ? io->win_gamma : nullptr, io->y};
  int buf = 0;
  if (dual1_tc_supported(g) && dual1_tc_inputs_ok(gio)) {
    // depth 1 on the tensor cores: every chunk's gate coefficients, then one
    // persistent launch that keeps the state on chip (it reads the raw keys,
    // queries, values and Omega weights itself)
    CUDA_TRY(dual1_coef_launch(g, gio, w.gpart, coef_layout_tc(g), st));
    buf = (g.T / g.C) & 1;
    CUDA_TRY(dual1_tc_launch(g, w, gio, w.gpart, buf, st));
    nl += 2;
  } else {
    CUDA_TRY(generic_prepare(g, w, gio, st, &nl));
    for (int s = 0; s < g.T; s += g.C) {
      const Chunk ch = dual1_chunk_at(g, s);
      CUDA_TRY(generic_chunk(g, ch, w, gio, buf, st, &nl));
      buf ^= 1;
    }
  }
  for (int m = 0; m < g.nmat; ++m) {
    const size_t bytes = (size_t)g.units * g.rows[m] * g.cols[m] * sizeof(float);
    CUDA_TRY(cudaMemcpyAsync(io->W_out[m], w.Wst[buf][m], bytes, cudaMemcpyDeviceToDevice, st));
    if (ns_tc) CUDA_TRY(ns_tc_state_out(g, m, w.Sst[buf][m], io->S_out[m], st));
    else CUDA_TRY(cudaMemcpyAsync(io->S_out[m], w.Sst[buf][m], bytes, cudaMemcpyDeviceToDevice, st));
  }
  if (g.c > 1 && (io->win_k_out || io->win_v_out || io->win_gamma_out))
    CUDA_TRY(generic_cache_out(g, gio, cache_tmp, io->win_k_out, io->win_v_out, io->win_gamma_out, st, &nl));
  *nl_out = nl;
  return ATLAS_OK;
}

static bool graphs_enabled() {
  const char* e = getenv("ATLAS_NO_GRAPH");
  return !(e && e[0] == '1');
}

extern "C" int atlas_mem_forward(atlas_mem_handle* h, const atlas_mem_io* io, void* stream) {
  if (!h) return ATLAS_ERR_INVALID_ARG;
  int rc = check_io(h, io);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  Geom g = h->base;
  g.units = io->B * io->H;
  g.T = io->T;
  g.n_prev = io->win_len;
  g.L = g.n_prev + g.T;
  const Layout L = layout(g, g.units, g.T);
  rc = ensure_workspace(h, L.total);
  if (rc) return rc;
  float* cache_tmp = nullptr;
  Work w = work_from(g, h->ws, L, &cache_tmp);
  h->status = w.status;
  if (mlp_tc_supported(g)) {
    // fused tensor-core kernel: state in/out and read-out in one launch
    CUDA_TRY(mlp_tc_launch(g, io->q, io->k, io->v, io->theta, io->eta, io->alpha, io->gamma, io->W0, io->S0, io->y,
                           io->W_out, io->S_out, w.status, st));
    h->launches = 1;
    h->last_stream = st;
    h->launched = true;
    return ATLAS_OK;
  }
  int nl = 0;
  if (graphs_enabled()) {
    const bool same_as_graph = h->gexec && h->gws == h->ws && memcmp(&h->gkey, io, sizeof *io) == 0;
    if (same_as_graph) {
      CUDA_TRY(cudaGraphLaunch(h->gexec, st));
      h->launches = h->glaunches;
      h->last_stream = st;
      h->launched = true;
      return ATLAS_OK;
    }
    const bool repeat = h->have_last && h->last_ws == h->ws && memcmp(&h->last_io, io, sizeof *io) == 0;
    h->last_io = *io;
    h->last_ws = h->ws;
    h->have_last = true;
    if (repeat) {
      if (!h->cap) CUDA_TRY(cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking));
      CUDA_TRY(cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal));
      const int rc2 = run_generic(h, g, w, io, cache_tmp, h->cap, &nl);
      cudaGraph_t graph = nullptr;
      const cudaError_t ec = cudaStreamEndCapture(h->cap, &graph);
      if (rc2) {
        if (graph) cudaGraphDestroy(graph);
        return rc2;
      }
      if (ec != cudaSuccess) return fail(h, ATLAS_ERR_CUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(ec));
      cudaGraphExec_t ex = nullptr;
      const cudaError_t ei = cudaGraphInstantiate(&ex, graph, 0);
      cudaGraphDestroy(graph);
      if (ei != cudaSuccess) return fail(h, ATLAS_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(ei));
      if (h->gexec) cudaGraphExecDestroy(h->gexec);
      h->gexec = ex;
      h->gkey = *io;
      h->gws = h->ws;
      h->glaunches = nl;
      CUDA_TRY(cudaGraphLaunch(h->gexec, st));
      h->launches = nl;
      h->last_stream = st;
      h->launched = true;
      return ATLAS_OK;
    }
  }
  rc = run_generic(h, g, w, io, cache_tmp, st, &nl);
  if (rc) return rc;
  h->launches = nl;
  h->last_stream = st;
  h->launched = true;
  return ATLAS_OK;
}

extern "C" int atlas_mem_status(atlas_mem_handle* h) {
  if (!h) return ATLAS_ERR_INVALID_ARG;
  if (!h->launched || !h->status) return ATLAS_OK;
  CUDA_TRY(cudaStreamSynchronize(h->last_stream));
  int s = 0;
  CUDA_TRY(cudaMemcpy(&s, h->status, sizeof s, cudaMemcpyDeviceToHost));
  if (s != 0) {
    CUDA_TRY(cudaMemset(h->status, 0, sizeof s));
    if (s == ATLAS_ERR_RANGE)
      return fail(h, ATLAS_ERR_RANGE,
                  "the fused kernel produced a non-finite y or state (an input beyond the range of its fp16 "
                  "operands, or a diverging memory): this call's outputs are not valid");
    return fail(h, ATLAS_ERR_TIMEOUT, "a device-side wait gave up (status %d)", s);
  }
  return ATLAS_OK;
}

struct Item {
  const void* src;   // host source of an input, else nullptr
  void* dst_host;    // host destination of an output, else nullptr
  size_t bytes;
};

// Host-buffer forward on the fused path, pipelined over time segments: the
// sequence is cut into NS segments of whole chunks; segment i's inputs are
// copied in on one stream while segment i-1 runs, the kernel runs segment i
// from the state segment i-1 left (fp32, so the result equals one launch
// bit for bit), and its y is copied out on a third stream while segment
// i+1 runs.  items / dptr follow the order of atlas_mem_forward_host
// (inputs q k v theta eta alpha gamma P W0[2] S0[2] window[3], then outputs
// y W_out[2] S_out[2] window[3]).
static int forward_host_pipelined(atlas_mem_handle* h, const atlas_mem_io* io, const Geom& g, const Item* items,
                                  void* const* dptr, int n, cudaStream_t st) {
  const int NS = atlas_mem_handle::kGroups;
  const size_t U = (size_t)g.units, T = (size_t)g.T, Ts = T / NS;
  const Layout L = layout(g, g.units, g.T);
  int rc = ensure_workspace(h, L.total);
  if (rc) return rc;
  float* cache_tmp = nullptr;
  Work w = work_from(g, h->ws, L, &cache_tmp);
  h->status = w.status;
  for (int i = 0; i < 2; ++i)
    if (!h->pst[i]) CUDA_TRY(cudaStreamCreateWithFlags(&h->pst[i], cudaStreamNonBlocking));
  for (int i = 0; i < 2 * NS + 2; ++i)
    if (!h->pev[i]) CUDA_TRY(cudaEventCreateWithFlags(&h->pev[i], cudaEventDisableTiming));
  cudaStream_t cin = h->pst[0], cout = h->pst[1];
  cudaEvent_t* in_done = h->pev;          // [NS]
  cudaEvent_t* k_done = h->pev + NS;      // [NS]
  cudaEvent_t start = h->pev[2 * NS], out_done = h->pev[2 * NS + 1];
  CUDA_TRY(cudaEventRecord(start, st));
  CUDA_TRY(cudaStreamWaitEvent(cin, start, 0));
  CUDA_TRY(cudaStreamWaitEvent(cout, start, 0));
  // one time segment of a [U][T][width] array: U rows of Ts * width bytes
  auto seg_copy = [&](int i, void* dst, const void* src, size_t bytes_per_unit, cudaMemcpyKind kind,
                      cudaStream_t s) -> cudaError_t {
    const size_t pitch = bytes_per_unit, wb = bytes_per_unit / NS, off = (size_t)i * wb;
    return cudaMemcpy2DAsync((char*)dst + off, pitch, (const char*)src + off, pitch, wb, U, kind, s);
  };
  // state in (whole), then each segment's per-token inputs
  for (int m = 8; m < 12; ++m)
    if (items[m].src && items[m].bytes)
      CUDA_TRY(cudaMemcpyAsync(dptr[m], items[m].src, items[m].bytes, cudaMemcpyHostToDevice, cin));
  const int per_token[] = {0, 1, 2, 3, 4, 5, 6};
  for (int i = 0; i < NS; ++i) {
    for (int a : per_token)
      if (items[a].src && items[a].bytes)
        CUDA_TRY(seg_copy(i, dptr[a], items[a].src, items[a].bytes / U, cudaMemcpyHostToDevice, cin));
    CUDA_TRY(cudaEventRecord(in_done[i], cin));
  }
  Geom gs = g;
  gs.T = (int)Ts;
  // the state ping-pongs between the staging of W0/S0 and of W_out/S_out
  float* st_a[4] = {(float*)dptr[8], (float*)dptr[9], (float*)dptr[10], (float*)dptr[11]};
  float* st_b[4] = {(float*)dptr[16], (float*)dptr[17], (float*)dptr[18], (float*)dptr[19]};
  const size_t es = g.qkv_dtype == ATLAS_BF16 ? 2 : 4;
  for (int i = 0; i < NS; ++i) {
    CUDA_TRY(cudaStreamWaitEvent(st, in_done[i], 0));
    float** sin = (i % 2 == 0) ? st_a : st_b;
    float** sout = (i % 2 == 0) ? st_b : st_a;
    const size_t t0 = (size_t)i * Ts;
    const char* q = (const char*)dptr[0] + t0 * g.d_k * es;
    const char* k = (const char*)dptr[1] + t0 * g.d_k * es;
    const char* v = (const char*)dptr[2] + t0 * g.d_v * es;
    const float* th = (const float*)dptr[3] + t0;
    const float* et = (const float*)dptr[4] + t0;
    const float* al = (const float*)dptr[5] + t0;
    const float* ga = dptr[6] ? (const float*)dptr[6] + t0 : nullptr;
    const float* W0[2] = {sin[0], sin[1]};
    const float* S0[2] = {sin[2], sin[3]};
    float* Wo[2] = {sout[0], sout[1]};
    float* So[2] = {sout[2], sout[3]};
    CUDA_TRY(mlp_tc_launch(gs, q, k, v, th, et, al, ga, W0, S0, (float*)dptr[15] + t0 * g.d_v, Wo, So, w.status, st,
                           (int)T));
    CUDA_TRY(cudaEventRecord(k_done[i], st));
    CUDA_TRY(cudaStreamWaitEvent(cout, k_done[i], 0));
    CUDA_TRY(seg_copy(i, items[15].dst_host, dptr[15], items[15].bytes / U, cudaMemcpyDeviceToHost, cout));
  }
  // final state: in st_b after an odd number of segments, else st_a
  float** fin = (NS % 2 == 1) ? st_b : st_a;
  for (int m = 0; m < 4; ++m)
    if (items[16 + m].dst_host && items[16 + m].bytes)
      CUDA_TRY(cudaMemcpyAsync(items[16 + m].dst_host, fin[m], items[16 + m].bytes, cudaMemcpyDeviceToHost, cout));
  CUDA_TRY(cudaEventRecord(out_done, cout));
  CUDA_TRY(cudaStreamWaitEvent(st, out_done, 0));
  h->launches = NS;
  h->last_stream = st;
  h->launched = true;
  (void)n;
  CUDA_TRY(cudaStreamSynchronize(st));
  return atlas_mem_status(h);
}

extern "C" int atlas_mem_forward_host(atlas_mem_handle* h, const atlas_mem_io* io, void* stream) {
  if (!h) return ATLAS_ERR_INVALID_ARG;
  int rc = check_io(h, io);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const Geom& g = h->base;
  const size_t U = (size_t)io->B * io->H, T = io->T;
  const size_t es = g.qkv_dtype == ATLAS_BF16 ? 2 : 4;
  const size_t ncache = (size_t)(g.c > 1 ? g.c - 1 : 0);
  // staged arrays: host source (input) or destination (output), bytes
  Item items[24];
  int n = 0;
  auto in = [&](const void* p, size_t bytes) { items[n++] = Item{p, nullptr, p ? bytes : 0}; };
  auto out = [&](void* p, size_t bytes) { items[n++] = Item{nullptr, p, p ? bytes : 0}; };
  in(io->q, U * T * g.d_k * es);
  in(io->k, U * T * g.d_k * es);
  in(io->v, U * T * g.d_v * es);
  in(io->theta, U * T * 4);
  in(io->eta, U * T * 4);
  in(io->alpha, U * T * 4);
  in(io->gamma, U * T * 4);
  in(io->P, (size_t)g.poly * g.proj_dim * es);
  for (int m = 0; m < 2; ++m) in(m < g.nmat ? io->W0[m] : nullptr, U * g.rows[m] * g.cols[m] * 4);
  for (int m = 0; m < 2; ++m) in(m < g.nmat ? io->S0[m] : nullptr, U * g.rows[m] * g.cols[m] * 4);
  in(io->win_len ? io->win_k : nullptr, U * ncache * g.d_k * es);
  in(io->win_len ? io->win_v : nullptr, U * ncache * g.d_v * es);
  in(io->win_len ? io->win_gamma : nullptr, U * ncache * 4);
  out(io->y, U * T * g.d_v * 4);
  for (int m = 0; m < 2; ++m) out(m < g.nmat ? io->W_out[m] : nullptr, U * g.rows[m] * g.cols[m] * 4);
  for (int m = 0; m < 2; ++m) out(m < g.nmat ? io->S_out[m] : nullptr, U * g.rows[m] * g.cols[m] * 4);
  out(g.c > 1 ? io->win_k_out : nullptr, U * ncache * g.d_k * es);
  out(g.c > 1 ? io->win_v_out : nullptr, U * ncache * g.d_v * es);
  out(g.c > 1 ? io->win_gamma_out : nullptr, U * ncache * 4);
  size_t off[24], total = 0;
  for (int i = 0; i < n; ++i) {
    off[i] = total;
    total += al(items[i].bytes);
  }
  if (h->stage_bytes < total) {
    if (h->stage) {
      CUDA_TRY(cudaDeviceSynchronize());
      cudaFree(h->stage);
      h->stage = nullptr;
      h->stage_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&h->stage, total);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(h, ATLAS_ERR_OOM, "staging cudaMalloc(%zu): %s", total, cudaGetErrorString(e));
    }
    h->stage_bytes = total;
  }
  char* base = (char*)h->stage;
  void* dptr[24];
  for (int i = 0; i < n; ++i) dptr[i] = items[i].bytes ? base + off[i] : nullptr;
  // fused path: pipeline over unit groups (every array but P is unit-major)
  Geom gu = g;
  gu.units = (int)U;
  gu.T = (int)T;
  gu.n_prev = io->win_len;
  gu.L = gu.n_prev + gu.T;
  const int NG = atlas_mem_handle::kGroups;
  if (mlp_tc_supported(gu) && io->P == nullptr && T % ((size_t)NG * g.C) == 0 &&
      getenv("ATLAS_NO_PIPELINE") == nullptr)
    return forward_host_pipelined(h, io, gu, items, dptr, n, st);
  for (int i = 0; i < n; ++i)
    if (items[i].src && items[i].bytes)
      CUDA_TRY(cudaMemcpyAsync(dptr[i], items[i].src, items[i].bytes, cudaMemcpyHostToDevice, st));
  atlas_mem_io d = *io;
  int i = 0;
  d.q = dptr[i++]; d.k = dptr[i++]; d.v = dptr[i++];
  d.theta = (const float*)dptr[i++]; d.eta = (const float*)dptr[i++]; d.alpha = (const float*)dptr[i++];
  d.gamma = (const float*)dptr[i++];
  d.P = dptr[i++];
  for (int m = 0; m < 2; ++m) d.W0[m] = (const float*)dptr[i++];
  for (int m = 0; m < 2; ++m) d.S0[m] = (const float*)dptr[i++];
  d.win_k = dptr[i++]; d.win_v = dptr[i++]; d.win_gamma = (const float*)dptr[i++];
  const int first_out = i;
  d.y = (float*)dptr[i++];
  for (int m = 0; m < 2; ++m) d.W_out[m] = (float*)dptr[i++];
  for (int m = 0; m < 2; ++m) d.S_out[m] = (float*)dptr[i++];
  d.win_k_out = dptr[i++]; d.win_v_out = dptr[i++]; d.win_gamma_out = (float*)dptr[i++];
  rc = atlas_mem_forward(h, &d, stream);
  if (rc) return rc;
  for (int j = first_out; j < n; ++j)
    if (items[j].dst_host && items[j].bytes)
      CUDA_TRY(cudaMemcpyAsync(items[j].dst_host, dptr[j], items[j].bytes, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  return atlas_mem_status(h);
}

// -------------------------------------------------- no-allocation variant
// Scratch for atlas_mem_forward_noalloc: a fixed device array, so that the
// entry point never allocates.  Every GPU that loads this library holds it
// until the process exits.  In host code this name is only a stand-in: the
// kernels get the device address from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATLAS_NOALLOC_SCRATCH_BYTES];

// The array's device address, looked up on every call with the calling
// device current (cheap, allocates nothing): an address cached across calls
// would go stale after a device reset or a new primary context.
static int noalloc_scratch(atlas_mem_handle* h, void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    int dev = -1;
    cudaGetDevice(&dev);
    return fail(h, ATLAS_ERR_CUDA, "cudaGetSymbolAddress(fixed scratch) on device %d: %s", dev,
                cudaGetErrorString(e));
  }
  *out = p;
  return ATLAS_OK;
}

extern "C" int atlas_mem_forward_noalloc(atlas_mem_handle* h, const atlas_mem_io* io, void* stream) {
  if (!h) return ATLAS_ERR_INVALID_ARG;
  int rc = check_io(h, io);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  Geom g = h->base;
  g.units = io->B * io->H;
  g.T = io->T;
  g.n_prev = io->win_len;
  g.L = g.n_prev + g.T;
  const Layout L = layout(g, g.units, g.T);
  const bool fused = mlp_tc_supported(g);
  // the fused kernel keeps its state on chip and needs only the status word;
  // the multi-launch path needs its whole working set in the array
  if (!fused && L.total > (size_t)ATLAS_NOALLOC_SCRATCH_BYTES)
    return fail(h, ATLAS_ERR_UNSUPPORTED,
                "this call needs %zu bytes of scratch but atlas_mem_forward_noalloc has a fixed %zu bytes; "
                "use fewer units or tokens per call, or atlas_mem_forward",
                L.total, (size_t)ATLAS_NOALLOC_SCRATCH_BYTES);
  void* base = nullptr;
  rc = noalloc_scratch(h, &base);
  if (rc) return rc;
  if (fused) {
    int* status = (int*)base;
    // the array keeps the previous call's contents: the status word must start at 0
    CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    h->status = status;
    CUDA_TRY(mlp_tc_launch(g, io->q, io->k, io->v, io->theta, io->eta, io->alpha, io->gamma, io->W0, io->S0, io->y,
                           io->W_out, io->S_out, status, st));
    h->launches = 1;
    h->last_stream = st;
    h->launched = true;
    return ATLAS_OK;
  }
  float* cache_tmp = nullptr;
  Work w = work_from(g, base, L, &cache_tmp);
  CUDA_TRY(cudaMemsetAsync(w.status, 0, sizeof(int), st));
  h->status = w.status;
  int nl = 0;
  rc = run_generic(h, g, w, io, cache_tmp, st, &nl);
  if (rc) return rc;
  h->launches = nl;
  h->last_stream = st;
  h->launched = true;
  return ATLAS_OK;
}
