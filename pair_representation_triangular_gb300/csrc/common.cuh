// Shared declarations of the CUDA library: the handle, device error codes and
// the kernel launchers of each path.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/tri_attn.h"

// Codes written into the handle's device error word (bitwise OR of causes).
#define TRI_DEV_ERR_TIMEOUT 1u
#define TRI_DEV_ERR_CHECK 2u

// Default cap of a bounded spin-wait, in polls (each poll is a try_wait with a
// hardware suspend hint, so this is on the order of a second).
#define TRI_DEFAULT_WAIT_LIMIT (1ll << 24)

// Split of the `mode` argument: the mask reading and the node variant.
inline bool tri_mode_valid(int mode) {
  return (mode & ~(TRI_ATTN_MASK_QUERY_KEY | TRI_ATTN_ENDING_NODE)) == 0;
}
inline int tri_mask_mode(int mode) { return mode & TRI_ATTN_MASK_QUERY_KEY; }
inline bool tri_ending(int mode) { return (mode & TRI_ATTN_ENDING_NODE) != 0; }

struct tri_attn_s {
  int B, N, D, h, d, dtype, mask_mode;
  bool ending;                     // ending-node variant (attention along columns)
  bool simt;                       // fp32 SIMT kernels (fp32 handles)
  long long cells;                 // B * N * N
  int device;
  // Packed weights (owned).
  void* w_proj;                    // f32: [D][4D+h] (in, out); bf16: [n_proj_pad][D] (out, in)
  void* w_out;                     // f32: [D][D] (in, out);    bf16: [D][D] (out, in)
  float* gamma; float* beta; float* bg; float* bo;   // fp32 copies
  float* wb_f32;                   // bf16 path: Wb as fp32 [h][D]
  // Workspace (owned).
  void* q; void* k; void* v; void* g; void* o;       // [cells][D], handle dtype
  float* bias;                     // [B][h][N][N]
  unsigned int* dev_err;           // device error word
  long long wait_limit;
  // Host-buffer staging (forward_host), allocated on first use.
  void* stage_x; int32_t* stage_mask; void* stage_out;
  // Tensor-core path state (opaque to the f32 path).
  void* tc;
  size_t bytes_owned;
  // Optional per-kernel timing: events recorded around each kernel of a forward.
  int timing;
  int n_marks;
  cudaEvent_t marks[8];
  const char* mark_names[8];
};

// Record timing mark `idx` (0 = before the first kernel; idx > 0 = after the
// kernel named `name`) when kernel timing is enabled on the handle.
inline void tri_mark(tri_attn_s* t, cudaStream_t s, int idx, const char* name) {
  if (!t->timing || idx >= 8) return;
  cudaEventRecord(t->marks[idx], s);
  t->mark_names[idx] = name;
  t->n_marks = idx + 1;
}

size_t tri_elem_size(int dtype);

// ---- fp32 SIMT path (kernels_f32.cu)
cudaError_t tri_f32_pack_weights(tri_attn_s* t, const void* Wq, const void* Wk, const void* Wv,
                                 const void* Wg, const void* Wb, const void* Wo,
                                 cudaStream_t s);
cudaError_t tri_f32_forward(tri_attn_s* t, cudaStream_t s, const float* x,
                            const int32_t* mask, float* out);

// fp32 forward on caller-provided buffers (no handle): weights in nn.Linear
// layout are packed into w_proj / w_out, intermediates go to q..o and bias.
struct TriF32Raw {
  int B, N, D, h, mask_mode;
  bool ending;
  const float *gamma, *beta, *Wq, *Wk, *Wv, *Wg, *bg, *Wb, *Wo, *bo;
  const float* x;
  const int32_t* mask;
  float* out;
  float *w_proj, *w_out, *q, *k, *v, *g, *o, *bias;
};
cudaError_t tri_f32_forward_raw(const TriF32Raw& a, cudaStream_t s);

// ---- bf16 tensor-core path (kernels_tc.cu; kernels in tc_k1.cu, tc_k2.cu, tc_k3.cu)
bool tri_tc_supported(int B, int N, int D, int h);
cudaError_t tri_tc_init(tri_attn_s* t, const void* Wq, const void* Wk, const void* Wv,
                        const void* Wg, const void* Wb, const void* Wo, cudaStream_t s);
void tri_tc_release(tri_attn_s* t);
cudaError_t tri_tc_forward(tri_attn_s* t, cudaStream_t s, const void* x,
                           const int32_t* mask, void* out);
// Host buffers xh, maskh, outh through the device staging buffers dx, dmask,
// dout, with the copies overlapped with the first and last kernels; queued on s.
cudaError_t tri_tc_forward_host(tri_attn_s* t, cudaStream_t s, const void* xh,
                                const int32_t* maskh, void* outh, void* dx, int32_t* dmask,
                                void* dout);
size_t tri_tc_extra_bytes(int B, int N, int D, int h);
int tri_tc_bias_row_stride(const tri_attn_s* t);
