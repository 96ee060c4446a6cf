/*
 * atlas_prologue.h -- C ABI of the stage in front of the Titans/ATLAS memory:
 * from the model-width sequence x to the memory's inputs q, k, v and its
 * gates.
 *
 * What it computes, for every batch row b and token t (row vectors):
 *   u_t = x_t W_in: one projection whose N columns are, in order, the query
 *       heads (H * d_k), the key heads (H * d_k), the value heads (H * d_v)
 *       and G * H gate logits, gate-major (theta heads, eta heads, alpha
 *       heads, then gamma heads when with_gamma); titans-torch 0.1.2 project
 *       page, API Reference (TitansMAC forward flow, q = W_Q S).
 *   The Nc = H (2 d_k + d_v) q/k/v channels pass a causal depthwise
 *       convolution of K = conv taps, no bias: conv_t[c] = sum_{j<K}
 *       conv_w[c][K-1-j] u_{t-j}[c] (atlas-torch README, "Atlas
 *       Extensions": CausalDepthwiseConv1d, kernel 4, on keys, values and
 *       queries).  Rows before the call come from the carried cache, else
 *       are zero.
 *   q and k of every head are divided by their L2 norm (by 1e-12 when the
 *       norm is smaller, so a zero vector stays zero); v is not normalised.
 *   theta = theta_max * sigmoid(l + b), eta, alpha (and gamma) = sigmoid(l +
 *       b), with l the head's logit column and b its bias (titans-torch
 *       0.1.2 project page, API Reference: the gates come from the data).
 *
 * The outputs have exactly the layouts atlas_mem_forward takes (atlas_mem.h),
 * so the two calls chain on one stream.
 *
 * Execution: asynchronous on the given CUDA stream; the projection is one
 * GEMM of the library's own (fp32 accumulation) into the handle's workspace:
 * for bf16 inputs tcgen05 tensor-core tiles fed by TMA, exact bf16 products;
 * for fp32 inputs, or strides and addresses TMA cannot take (D or N not a
 * multiple of 8, x or W_in not 16-byte aligned), an fp32 SIMT GEMM.  The
 * rest is one kernel.  A handle is not re-entrant across concurrent
 * streams.
 *
 * Errors: the status codes of atlas_mem.h; atlas_prologue_last_error gives
 * the message.  Validation failures return before any CUDA call.
 */
#ifndef ATLAS_PROLOGUE_H
#define ATLAS_PROLOGUE_H

#include <stddef.h>

#include "atlas_mem.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int D;            /* model width of x (>= 1) */
    int H;            /* heads (>= 1) */
    int d_k, d_v;     /* head widths of q/k and of v (2 d_k + d_v <= 512) */
    int conv;         /* taps K of the causal depthwise convolution, 1..8 (1 = none) */
    int with_gamma;   /* 1: a fourth gate head gives the Omega weights gamma */
    float theta_max;  /* theta = theta_max * sigmoid(.), > 0 */
    int qkv_dtype;    /* ATLAS_F32 or ATLAS_BF16: type of x, W_in and q, k, v */
} atlas_prologue_config;

typedef struct atlas_prologue_handle atlas_prologue_handle;

/*
 * Tensors of one call, all DEVICE pointers owned by the caller.  N = Nc +
 * G H with Nc = H (2 d_k + d_v) and G = 3 + with_gamma.
 */
typedef struct {
    int B, T;                 /* B >= 1, T >= 1 */
    const void* x;            /* [B][T][D]  qkv_dtype */
    const void* W_in;         /* [D][N]     qkv_dtype, row-major */
    const float* conv_w;      /* [Nc][conv] taps; tap conv-1 weighs the current token */
    const float* gate_b;      /* [G][H] biases of the gate heads */
    const float* cache;       /* NULL (sequence start) or [B][conv-1][Nc]: the projected
                               * q/k/v rows of the conv-1 tokens before this call, oldest first */
    void* q;                  /* [B][H][T][d_k] qkv_dtype (bf16: round to nearest even) */
    void* k;                  /* [B][H][T][d_k] qkv_dtype */
    void* v;                  /* [B][H][T][d_v] qkv_dtype */
    float* theta;             /* [B][H][T] */
    float* eta;               /* [B][H][T] */
    float* alpha;             /* [B][H][T] */
    float* gamma;             /* [B][H][T] with with_gamma, else must be NULL */
    float* cache_out;         /* NULL or [B][conv-1][Nc]: the cache for the next call;
                               * must not alias cache */
} atlas_prologue_io;

/* Validate the config and make a handle (no CUDA call).  INVALID_ARG or
 * UNSUPPORTED with a message from atlas_prologue_last_error(NULL). */
int atlas_prologue_create(const atlas_prologue_config* cfg, atlas_prologue_handle** out);

/* One call; stream is a cudaStream_t (NULL = the default stream).  Grows the
 * handle's workspace to atlas_prologue_workspace_bytes on first use. */
int atlas_prologue_forward(atlas_prologue_handle* h, const atlas_prologue_io* io, void* stream);

/* Device workspace a call of this size needs: the fp32 projection, B T N floats. */
size_t atlas_prologue_workspace_bytes(const atlas_prologue_handle* h, int B, int T);

/* Wait for the last forward on h and return its device status: ATLAS_OK, or
 * ATLAS_ERR_TIMEOUT if a bounded wait of the tensor-core projection gave up
 * (its outputs are then not valid).  Clears the status word. */
int atlas_prologue_status(atlas_prologue_handle* h);

/* Which projection GEMM the last forward on h ran: 1 = tensor cores (TMA +
 * tcgen05), 0 = fp32 SIMT, -1 = none yet. */
int atlas_prologue_last_gemm(const atlas_prologue_handle* h);

/* Message of the last failure on h, or of the last failed create when h is NULL. */
const char* atlas_prologue_last_error(const atlas_prologue_handle* h);

/* Free the handle and its workspace (NULL is a no-op). */
void atlas_prologue_destroy(atlas_prologue_handle* h);

#ifdef __cplusplus
}
#endif

#endif
