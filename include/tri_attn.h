/*
 * tri_attn.h -- C ABI of libtriattn: the forward pass of starting-node
 * triangular self-attention over a pair representation, on one GB300 GPU.
 *
 * Operation (POPCORNBENCH "Kimi-K2.6 l2_p6", forward op list steps 1-18, and
 * "FW-GLM-5-1 l2_p6", the quoted reference Model.forward), for each cell
 * (b, r, c) of the B x N x N pair grid with D channels, h heads, d = D / h:
 *
 *   x_hat = LayerNorm(pair_repr[b,r,c,:])            (eps 1e-5, biased variance)
 *   q, k, v = Wq x_hat, Wk x_hat, Wv x_hat            (no bias)
 *   g = sigmoid(Wg x_hat + bg)
 *   bias[b,t,r,c] = (Wb x_hat)[t]                     (no bias; shared by all rows)
 *   for each row i, head t, query j:
 *     l_k = q[b,i,j,t].k[b,i,k,t] / sqrt(d) + bias[b,t,j,k]
 *     l_k = -1e9 where the mask drops key k           (replacement, not addition)
 *     o[b,i,j,t] = sum_k softmax_k(l) v[b,i,k,t]
 *   out[b,i,j,:] = Wo (g * o) + bo                    (dropout is the identity)
 *
 * Mask readings (the pages disagree; both are offered):
 *   TRI_ATTN_MASK_ROW_KEY   key k of row i is dropped when pair_mask[b,i,k] == 0
 *   TRI_ATTN_MASK_QUERY_KEY key k of query j is dropped when pair_mask[b,j,k] == 0
 *                           (the quoted code's broadcast of pair_mask over rows i)
 * A softmax row whose keys are all dropped gets the uniform weight 1/N.
 *
 * Node variants (OR-ed into the mask reading to form the `mode` argument):
 *   TRI_ATTN_STARTING_NODE  the operation above: attention along rows i.
 *   TRI_ATTN_ENDING_NODE    the same module on the grid with its two node axes
 *                           exchanged, out = T(f(T(pair_repr), T(pair_mask)))
 *                           where T swaps the two N axes; per output cell
 *                           (b, i, j) the softmax runs along column j:
 *       l_k = q[b,i,j,t].k[b,k,j,t] / sqrt(d) + bias[b,t,k,i]
 *       o[b,i,j,t] = sum_k softmax_k(l) v[b,k,j,t]
 *     with key k dropped when pair_mask[b,k,j] == 0 (row-key reading) or
 *     pair_mask[b,k,i] == 0 (query-key reading). The pages name only the
 *     starting-node module; this reading of its counterpart is the plainest one.
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major (C order), of the element type given by
 *     `dtype` (float for TRI_ATTN_F32, bfloat16 for TRI_ATTN_BF16); pair_mask is
 *     int32 with any nonzero entry meaning "keep". Linear weights use the
 *     nn.Linear layout (out_features, in_features).
 *   - Device pointers are addresses in the current CUDA context's device memory,
 *     16-byte aligned. `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - Status codes are returned; nothing aborts, throws or traps across the ABI.
 *     Errors detected on the device (a bounded wait that ran out, a failed
 *     bounds check) are recorded in the handle and reported by
 *     tri_attn_sync_check.
 *   - A handle may be used from one stream at a time: its workspace is shared
 *     by all calls.
 */
#ifndef TRI_ATTN_H
#define TRI_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tri_attn_s* tri_attn_t;

enum { TRI_ATTN_F32 = 0, TRI_ATTN_BF16 = 1 };
enum { TRI_ATTN_MASK_ROW_KEY = 0, TRI_ATTN_MASK_QUERY_KEY = 1 };
enum { TRI_ATTN_STARTING_NODE = 0, TRI_ATTN_ENDING_NODE = 2 };
enum { TRI_ATTN_PATH_SIMT = 0, TRI_ATTN_PATH_TENSOR_CORE = 1 };

enum {
  TRI_ATTN_OK = 0,
  TRI_ATTN_ERR_INVALID_ARG = 1,    /* bad pointer, shape, alignment or handle       */
  TRI_ATTN_ERR_UNSUPPORTED = 2,    /* valid but not built (e.g. bf16 with d = 128)  */
  TRI_ATTN_ERR_CUDA = 3,           /* a CUDA runtime call failed                     */
  TRI_ATTN_ERR_OOM = 4,            /* device allocation failed                       */
  TRI_ATTN_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait ran out                */
  TRI_ATTN_ERR_DEVICE_CHECK = 6    /* a kernel's own bounds/alignment check failed   */
};

/* Build a handle for one problem shape and one set of weights: the module's
 * constructor, ModelNew(pair_dim = D, num_heads = h, dropout) on
 * "Kimi-K2.6 l2_p6" (layer definitions), with the dropout of the inference
 * forward, the identity (no dropout argument).
 *
 * B, N, D, h: batch, pair-grid side, channels, heads; D % h == 0. Supported:
 *   TRI_ATTN_F32  any B, N >= 1, even D <= 256 with d = D/h <= 128, on the fp32
 *                 SIMT kernels;
 *   TRI_ATTN_BF16 the tensor-core kernels, for D in {32, 64, 128} and
 *                 d = D/h in {16, 32, 64} (D = 128, h = 4 among them), any B,
 *                 1 <= N <= 8192, B*N*N < 2^31.
 *   Other shapes return TRI_ATTN_ERR_UNSUPPORTED before any CUDA call: there is
 *   no second bf16 backend and nothing runs on the host.
 * mode: a mask reading (TRI_ATTN_MASK_ROW_KEY or TRI_ATTN_MASK_QUERY_KEY),
 *   OR-ed with TRI_ATTN_ENDING_NODE for the ending-node variant (see above);
 *   any other bit gives TRI_ATTN_ERR_INVALID_ARG.
 * Weights (device pointers, element type `dtype`), nn.Linear layout:
 *   ln_gamma, ln_beta [D]; Wq, Wk, Wv, Wg [D][D]; bg [D]; Wb [h][D]; Wo [D][D]; bo [D].
 *   Which Linear carries a bias follows the layer definitions on
 *   "Kimi-K2.6 l2_p6": gate and out_proj do; query, key, value and bias_proj
 *   do not.
 * The weights are copied and repacked into memory the handle owns, on `stream`,
 * and the call synchronises `stream` before returning, so the caller may free
 * its weight buffers afterwards. The handle also owns the workspace for the
 * intermediates (q, k, v, g, the bias plane and the attention output).
 * On success *out receives the handle; on failure *out is NULL and nothing
 * is leaked. */
int tri_attn_create(tri_attn_t* out, int B, int N, int D, int h, int dtype, int mode,
                    const void* ln_gamma, const void* ln_beta,
                    const void* Wq, const void* Wk, const void* Wv,
                    const void* Wg, const void* bg, const void* Wb,
                    const void* Wo, const void* bo, void* stream);

/* One forward pass, asynchronous on `stream`; allocates nothing. The module's
 * forward(pair_repr, pair_mask) on "Kimi-K2.6 l2_p6" (forward op list steps
 * 1-18; the mask broadcast as in the Model.forward quoted on
 * "FW-GLM-5-1 l2_p6"), computed as written at the top of this header.
 *
 * pair_repr: device (B, N, N, D) of the handle's dtype, 16-byte aligned.
 * pair_mask: device (B, N, N) int32, nonzero = keep.
 * out:       device (B, N, N, D) of the handle's dtype; must not overlap the inputs.
 * The inputs must stay valid until the stream work completes. Argument and
 * launch errors are returned at once; device-side errors surface through
 * tri_attn_sync_check. */
int tri_attn_forward(tri_attn_t t, void* stream, const void* pair_repr,
                     const int32_t* pair_mask, void* out);

/* The same forward pass on HOST buffers (the operation of tri_attn_forward;
 * the pages' forward takes tensors wherever they live, this call is the
 * host-memory form of it): copies pair_repr and pair_mask to the
 * device (into staging buffers the handle owns; allocated at the first call),
 * runs the forward pass and copies the result back into `out_host`, ordered
 * after the work already queued on `stream`, then synchronises `stream` and
 * reports device-side errors like tri_attn_sync_check. On the tensor-core path
 * the copies run on two internal streams in chunks, overlapped with the
 * kernels (rows of x in, finished lines of out back); the result is bit-for-bit
 * that of tri_attn_forward. Host buffers should be page-locked for full copy
 * speed; pageable memory works but copies synchronously. On an error return no
 * copy that touches the host buffers is still running. */
int tri_attn_forward_host(tri_attn_t t, void* stream, const void* pair_repr_host,
                          const int32_t* pair_mask_host, void* out_host);

/* Synchronise `stream`, then report any error the handle's kernels recorded on
 * the device since the last check (and clear it). The pages have no
 * counterpart: their module raises no device-side errors; this reports the
 * bounded waits and checks of this library's kernels. */
int tri_attn_sync_check(tri_attn_t t, void* stream);

/* Release everything the handle owns (the end of the module's lifetime; no
 * counterpart on the pages). The caller must make sure no work that uses the
 * handle is still running. NULL is accepted. */
int tri_attn_destroy(tri_attn_t t);

/* Which kernels a handle runs: TRI_ATTN_PATH_TENSOR_CORE for every bf16 handle,
 * TRI_ATTN_PATH_SIMT for every fp32 handle (negative status for a NULL handle).
 * No counterpart on the pages. */
int tri_attn_kernel_path(tri_attn_t t);

/* Human-readable name of a status code (static storage; no counterpart on the
 * pages). */
const char* tri_attn_status_string(int status);

/* Bytes of device memory a handle of this shape owns (weights + workspace); the
 * same shape rules and status codes as tri_attn_create, checked without any
 * CUDA call. No counterpart on the pages. */
int tri_attn_workspace_bytes(int B, int N, int D, int h, int dtype, size_t* bytes);

/* Per-kernel timing (instrumentation; no counterpart on the pages). With
 * `enable` nonzero, every later tri_attn_forward records a CUDA event on its
 * stream before its first kernel and after each kernel
 * (events the handle owns; a few microseconds of stream work per forward).
 * tri_attn_kernel_times then reports the duration of each kernel of the most
 * recent forward. */
int tri_attn_enable_kernel_timing(tri_attn_t t, int enable);

/* Durations (milliseconds) of the kernels of the most recent forward, in launch
 * order; waits for that forward to finish. On entry *n is the capacity of `ms`
 * (and of `names`, which may be NULL); on return it is the number of kernels
 * (0 when timing is off or nothing ran). names[i] receives a static string. */
int tri_attn_kernel_times(tri_attn_t t, float* ms, const char** names, int* n);

/* Diagnostic access to the handle's intermediates, the tensors of the forward
 * op list on "Kimi-K2.6 l2_p6" before the gate and output projection (valid
 * until destroy; they
 * hold the results of the most recent forward once it has finished):
 *   "q", "k", "v", "g", "o"  (B*N*N, D) per cell the projections, the
 *                           post-sigmoid gate and the attention output before
 *                           the gate: bf16 on the tensor-core path (q times
 *                           log2(e)/sqrt(d); v in fp16, times a power of 2
 *                           that is 1 unless the weights could drive |v| past
 *                           2^15), fp32 on the SIMT path;
 *   "bias"                  (B, h, N, row_stride) pair-bias plane indexed
 *                           [b, t, query, key]: bias[b,t,j,k] for the starting
 *                           node, bias[b,t,k,i] at [b,t,i,k] for the ending
 *                           node; fp32 on the SIMT path; on the tensor-core
 *                           path fp16 holding log2(e) * bias, and -inf where
 *                           the query-key mask drops the key.
 * Returns the device pointer, or NULL for an unknown name or handle;
 * *row_stride (may be NULL) receives the innermost row stride in elements. */
void* tri_attn_debug_tensor(tri_attn_t t, const char* name, int64_t* row_stride);

/* Test hook: cap every bounded device-side wait of this handle's kernels at
 * `spins` polls (0 restores the default of about one second). A cap of 1
 * makes the first wait that is not already complete give up, so the timeout
 * path can be exercised without hanging the GPU. */
int tri_attn_set_wait_limit(tri_attn_t t, long long spins);

/* fp32 forward pass that allocates no device memory. The pages have no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc when they need a forward pass (code running inside a memory pool
 * or custom allocator that forbids outside allocations, plugins that are handed
 * only their input and output buffers, loops where an allocation and the
 * synchronisation it may cause are not allowed), so they cannot use
 * tri_attn_create, which allocates its weights and workspace.
 *
 * Everything is a caller pointer (device, fp32, 16-byte aligned; pair_mask
 * int32): the weights in nn.Linear layout as for tri_attn_create, pair_repr
 * (B, N, N, D), pair_mask (B, N, N) and out (B, N, N, D). The intermediates live
 * in one fixed 16 MiB device array inside the library, which every device the
 * library's code is loaded on holds until the process exits. A problem needs
 *   4 * (P * D + D * D + 5 * B * N * N * D + B * h * N * N) bytes, P = 4D + h
 * rounded up to an even count (each of those seven regions rounded up to 256);
 * larger problems return TRI_ATTN_ERR_UNSUPPORTED without launching anything.
 * Other shape rules are those of TRI_ATTN_F32 in tri_attn_create; `mode` is as
 * there.
 *
 * The call is asynchronous on `stream`. CUDA loads a library's device code
 * lazily: the first call on each device (each context) loads it, which
 * reserves the 16 MiB array in device memory and may synchronise, so make that
 * first call before any stream capture and outside any region that forbids
 * allocations; later calls allocate nothing. Every call looks up the array's
 * device address in the current context (cudaGetSymbolAddress), so a context
 * that was reset or re-created is served at its own address. All calls share the one
 * array and it keeps the previous call's contents (every byte a call reads is
 * written earlier in the same call, so nothing is cleared): calls that can
 * overlap on the GPU, on different streams or from different threads, race on
 * it and must be serialised by the caller. */
int tri_attn_forward_noalloc(int B, int N, int D, int h, int mode,
                             const float* ln_gamma, const float* ln_beta,
                             const float* Wq, const float* Wk, const float* Wv,
                             const float* Wg, const float* bg, const float* Wb,
                             const float* Wo, const float* bo, void* stream,
                             const float* pair_repr, const int32_t* pair_mask, float* out);

#ifdef __cplusplus
}
#endif
#endif /* TRI_ATTN_H */
