/*
 * atlas_mem.h -- C ABI of the GB300 Titans/ATLAS neural-memory forward.
 *
 * The operation (per (batch, head) unit, token by token):
 *
 *   x_i = phi(k_i), r_t = phi(q_t)   phi = identity (p = 1) or the exact
 *        degree-2 monomial map [1, x_i, x_i x_j / 2 (i <= j)], optionally
 *        times a projection P        (atlas-torch README, "Atlas Extensions":
 *                                      Polynomial Features; ATLAS summary 3.1)
 *   M_W(x) = x W          (depth 1)  or  x + SiLU(x W1) W2  (depth 2)
 *                                     (titans-pytorch-mlx README, Key
 *                                      Innovations; ATLAS summary 5.1)
 *   g_t = sum_{i=max(t0,t-c+1)}^{t} gamma_i grad ||M_Wbar(x_i) - v_i||^2
 *        with Wbar the weights at the start of t's chunk of C tokens
 *                                     (titans-pytorch-mlx README Eq. 12;
 *                                      ATLAS summary 3.2, 3.3)
 *   S_t = eta_t S_{t-1} - theta_t g_t                            (Eq. 14)
 *   U_t = NS_k(S_t) per matrix (k Newton-Schulz steps) or S_t   (ATLAS 5)
 *   W_t = (1 - alpha_t) W_{t-1} + U_t                            (Eq. 13)
 *   y_t = M_{W_t}(r_t)   (post-update read-out; atlas-torch README,
 *                         "Known deviations from the paper's MAC")
 *
 * Everything is row-major.  "units" = B*H.  Matrix m of the memory has
 * shape rows_m x cols_m: depth 1: (F, d_v); depth 2: (F, hidden), (hidden, d_v)
 * with F = d_k (p = 1), (d_k+1)(d_k+2)/2 (p = 2) or proj_dim (projected).
 *
 * Errors: every entry point returns an ATLAS_* status; nothing throws.
 * atlas_mem_last_error() returns a message for the last failure on a handle.
 * A handle is not re-entrant: do not call it from two threads or on two
 * streams at once.
 */
#ifndef ATLAS_MEM_H
#define ATLAS_MEM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define ATLAS_OK 0
#define ATLAS_ERR_INVALID_ARG 1   /* null pointer, bad size, inconsistent config */
#define ATLAS_ERR_UNSUPPORTED 2   /* valid request outside what the kernels cover */
#define ATLAS_ERR_CUDA 3          /* a CUDA runtime call failed (message has the name) */
#define ATLAS_ERR_OOM 4           /* workspace allocation failed */
#define ATLAS_ERR_TIMEOUT 5       /* a device-side bounded wait gave up */
#define ATLAS_ERR_RANGE 6         /* the fused MLP kernel produced a non-finite y or final state:
                                     an input beyond the range of its fp16 operands (keys, queries
                                     or values far from unit scale) or a memory that diverged; the
                                     outputs of that call are not valid */

/* element types of q, k, v, P and the window cache */
#define ATLAS_F32 0
#define ATLAS_BF16 1

/* read-out modes (atlas_mem_config.readout) */
#define ATLAS_READOUT_POST 0
#define ATLAS_READOUT_PRE 1

/* where Newton-Schulz applies (atlas_mem_config.ns_target) */
#define ATLAS_NS_MOMENTUM 0
#define ATLAS_NS_SURPRISE 1

/* update rules (atlas_mem_config.update) */
#define ATLAS_UPDATE_PER_TOKEN 0
#define ATLAS_UPDATE_CHUNKWISE 1

typedef struct {
    int depth;      /* 1 (matrix memory) or 2 (residual SiLU MLP) */
    int d_k;        /* key/query width before the feature map */
    int d_v;        /* value width; depth 2 needs F == d_v (residual) */
    int hidden;     /* MLP hidden width (depth 2), else ignored */
    int C;          /* tokens per chunk (C + c - 1 <= 1024, else UNSUPPORTED);
                     * gradients use the chunk-start weights */
    int c;          /* Omega window: the last c tokens, including t (c >= 1) */
    int p;          /* polynomial degree of the feature map: 1 or 2 */
    int proj_dim;   /* 0: no projection; else features are x P, P [poly_dim, proj_dim] */
    int ns_iters;   /* Newton-Schulz steps applied to the momentum, 0 = off */
    int qkv_dtype;  /* ATLAS_F32 or ATLAS_BF16 (q, k, v, P, window cache) */
    int readout;    /* ATLAS_READOUT_POST: y_t = M_t(q_t), the memory after token t's
                     * update (atlas-torch README, "Known deviations from the
                     * paper's MAC"); ATLAS_READOUT_PRE: y_t = M_{t-1}(q_t), the
                     * memory before it (titans-pytorch-mlx README, MAC, Eq. 21).
                     * The state written back is the same either way. */
    int ns_target;  /* with ns_iters > 0: ATLAS_NS_MOMENTUM orthogonalises the
                     * applied momentum, U_t = NS(S_t) (ATLAS summary, Section
                     * 5); ATLAS_NS_SURPRISE orthogonalises each token's windowed
                     * gradient with eta and theta outside, S_t = eta_t S_{t-1}
                     * - theta_t NS(g_t), W_t = (1 - alpha_t) W_{t-1} + S_t
                     * (atlas-torch README, "Atlas Extensions": Muon / Newton-
                     * Schulz on the surprise; "eta outside Newton-Schulz").
                     * The surprise has rank <= c, so it needs c <= 32. */
    int update;     /* ATLAS_UPDATE_PER_TOKEN: the per-token rule above (a
                     * momentum, decay and read-out step for every token).
                     * ATLAS_UPDATE_CHUNKWISE: the titans-pytorch chunk-wise
                     * store path (atlas-torch README, "Bug Fixes": the
                     * per_token_updates flag): per chunk one gradient
                     * G = sum_i theta_i gamma_i grad l_i(W_bar) over its
                     * tokens, eta and alpha pooled to their mean over the
                     * chunk, S <- eta_bar S - G, W <- (1 - alpha_bar) W +
                     * NS(S) (or + S); token t reads the memory after the last
                     * chunk ending at or before t (READOUT_POST) or its
                     * chunk's start memory (READOUT_PRE).  Needs c == 1 and
                     * Newton-Schulz, if any, on the momentum. */
} atlas_mem_config;

typedef struct atlas_mem_handle atlas_mem_handle;

/*
 * Tensors of one forward call.  In atlas_mem_forward every pointer is a
 * DEVICE pointer; in atlas_mem_forward_host every pointer is a HOST pointer
 * (page-locked memory is faster but not required).  The caller owns all of
 * them.  Outputs may alias the matching inputs (W_out[m] == W0[m],
 * S_out[m] == S0[m], win_*_out == win_*) for in-place continuation.
 */
typedef struct {
    int B, H, T;                 /* T % C == 0 and T > 0 */
    const void* q;               /* [B,H,T,d_k]  qkv_dtype */
    const void* k;               /* [B,H,T,d_k]  qkv_dtype */
    const void* v;               /* [B,H,T,d_v]  qkv_dtype */
    const float* theta;          /* [B,H,T] step size  */
    const float* eta;            /* [B,H,T] momentum   */
    const float* alpha;          /* [B,H,T] decay      */
    const float* gamma;          /* [B,H,T] Omega weights; NULL means all 1 */
    const void* P;               /* [poly_dim, proj_dim] qkv_dtype; NULL iff proj_dim == 0 */
    const float* W0[2];          /* initial weights, matrix m: [B,H,rows_m,cols_m]; [1] unused at depth 1 */
    const float* S0[2];          /* initial momentum, same shapes */
    /* Omega window cache: the raw keys, values and weights of the tokens that
     * precede this call (c-1 slots per unit, right-aligned: the last win_len
     * slots are valid, oldest first).  win_len = 0 starts a sequence; the
     * pointers may then be NULL.  Needed only when c > 1. */
    int win_len;                 /* 0 <= win_len <= c-1 */
    const void* win_k;           /* [B,H,c-1,d_k] qkv_dtype */
    const void* win_v;           /* [B,H,c-1,d_v] qkv_dtype */
    const float* win_gamma;      /* [B,H,c-1] */
    float* y;                    /* [B,H,T,d_v] read-out */
    float* W_out[2];             /* final weights W_T, shapes as W0 */
    float* S_out[2];             /* final momentum S_T (not orthogonalised) */
    /* outgoing cache, right-aligned, min(c-1, win_len+T) valid slots;
     * may be NULL when c == 1 or when not wanted */
    void* win_k_out;
    void* win_v_out;
    float* win_gamma_out;
} atlas_mem_io;

/* Validate a config and create a handle.  Returns INVALID_ARG for sizes that
 * make no sense and UNSUPPORTED for shapes the kernels do not cover. */
int atlas_mem_create(const atlas_mem_config* cfg, atlas_mem_handle** out);

/* Run the forward on `stream` (a cudaStream_t; NULL = legacy default stream).
 * Asynchronous: returns after the launches are queued.  Device pointers only.
 * The first call with a new largest (B, H, T) allocates the handle's device
 * workspace (cudaMalloc, synchronous).  Device-side failures (a bounded wait
 * that ran out) are reported by atlas_mem_status(). */
int atlas_mem_forward(atlas_mem_handle* h, const atlas_mem_io* io, void* stream);

/* The same forward on HOST buffers: copies the inputs to the device
 * (cudaMemcpyAsync on `stream`), runs the forward, copies y, W_T, S_T and the
 * cache back and synchronises `stream` before returning. */
int atlas_mem_forward_host(atlas_mem_handle* h, const atlas_mem_io* io, void* stream);

/* Size of the fixed device scratch of atlas_mem_forward_noalloc: 16 MiB. */
#define ATLAS_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

/* atlas_mem_forward for callers that must not allocate device memory.
 *
 * No counterpart in the pages: this is a deployment variant.  Some hosts
 * cannot let a library call cudaMalloc: a framework whose pool allocator owns
 * the device memory (a raw cudaMalloc would fail or fragment its pool), or a
 * serving loop that forbids allocation after start-up because cudaMalloc may
 * synchronise the device and stall other streams.  This entry point runs the
 * same forward as atlas_mem_forward (same arguments, device pointers, same
 * kernels, so the same results bit for bit) but takes its working memory from
 * a fixed array of ATLAS_NOALLOC_SCRATCH_BYTES that lives in the library's
 * device image, and calls no cudaMalloc, cudaFree or allocating library
 * routine.  The caller still passes every input and output buffer.
 *
 * - Shapes the fused MLP kernel covers keep their whole state on chip and use
 *   only the array's status word: any B, H, T.
 * - Other calls whose working set exceeds the array
 *   (atlas_mem_workspace_bytes(h, B, H, T) > ATLAS_NOALLOC_SCRATCH_BYTES)
 *   return ATLAS_ERR_UNSUPPORTED with a message giving both sizes; nothing is
 *   launched.
 * - Every call looks up the array's device address (cudaGetSymbolAddress)
 *   with the calling device current, so the address is never stale after a
 *   device reset; the first lookup on a device may load the library's device
 *   code, so make the first call on each device before any stream capture.
 * - Every call, from every handle, shares the one array per device and finds
 *   the previous call's contents there (the status word is cleared on each
 *   call).  Calls whose work overlaps on the GPU race on it: serialise them
 *   (one stream, or events between streams).
 * - Every GPU that loads the library holds the array until the process exits. */
int atlas_mem_forward_noalloc(atlas_mem_handle* h, const atlas_mem_io* io, void* stream);

/* Wait for the last forward on this handle and return its device status
 * (ATLAS_OK, ATLAS_ERR_TIMEOUT or ATLAS_ERR_RANGE).  Clears the status word. */
int atlas_mem_status(atlas_mem_handle* h);

/* Device workspace, in bytes, that a forward of this size uses. */
size_t atlas_mem_workspace_bytes(const atlas_mem_handle* h, int B, int H, int T);

/* Number of CUDA kernels the last atlas_mem_forward on this handle launched
 * (copies excluded). */
int atlas_mem_last_launches(const atlas_mem_handle* h);

/* Message of the last failure on this handle ("" if none).  With h == NULL:
 * the message of the calling thread's last failed atlas_mem_create. */
const char* atlas_mem_last_error(const atlas_mem_handle* h);

void atlas_mem_destroy(atlas_mem_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* ATLAS_MEM_H */
