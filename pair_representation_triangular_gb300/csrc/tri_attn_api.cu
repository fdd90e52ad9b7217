// C ABI of libtriattn: argument checks, ownership of weights and workspace,
// dispatch by dtype: fp32 handles run the fp32 SIMT kernels, bf16 handles the
// tensor-core kernels (bf16 shapes those do not cover are refused at create).
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TRI_ATTN_OK;
  if (e == cudaErrorMemoryAllocation) return TRI_ATTN_ERR_OOM;
  return TRI_ATTN_ERR_CUDA;
}

// Convert n elements of `dtype` at src (device) to fp32 at dst (device).
__global__ void to_f32_kernel(const void* src, int dtype, int n, float* dst) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  dst[i] = dtype == TRI_ATTN_F32 ? ((const float*)src)[i]
                                 : __bfloat162float(((const __nv_bfloat16*)src)[i]);
}

cudaError_t to_f32(const void* src, int dtype, int n, float* dst, cudaStream_t s) {
  to_f32_kernel<<<(n + 255) / 256, 256, 0, s>>>(src, dtype, n, dst);
  return cudaGetLastError();
}

// Shapes the fp32 SIMT kernels take: even D <= 256, d <= 128.
bool simt_shape(int D, int h) { return D <= 256 && D / h <= 128 && !(D & 1); }

void free_all(tri_attn_s* t) {
  if (!t) return;
  if (t->tc) tri_tc_release(t);
  if (t->timing)
    for (int i = 0; i < 8; ++i) cudaEventDestroy(t->marks[i]);
  void* ptrs[] = {t->w_proj, t->w_out, t->gamma, t->beta, t->bg, t->bo, t->wb_f32,
                  t->q, t->k, t->v, t->g, t->o, t->bias, t->dev_err,
                  t->stage_x, t->stage_mask, t->stage_out};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  free(t);
}

int check_shape(int B, int N, int D, int h, int dtype) {
  if (B < 1 || N < 1 || D < 1 || h < 1 || D % h) return TRI_ATTN_ERR_INVALID_ARG;
  if (dtype != TRI_ATTN_F32 && dtype != TRI_ATTN_BF16) return TRI_ATTN_ERR_INVALID_ARG;
  const long long cells = (long long)B * N * N;
  if (cells * (long long)D > (1ll << 40)) return TRI_ATTN_ERR_INVALID_ARG;
  // bf16 runs on the tensor-core kernels alone: D in {32, 64, 128} and
  // d = D / h in {16, 32, 64}, with B N^2 below 2^31 cells; there is no other
  // bf16 backend.
  if (dtype == TRI_ATTN_F32 ? !simt_shape(D, h) : !tri_tc_supported(B, N, D, h))
    return TRI_ATTN_ERR_UNSUPPORTED;
  return TRI_ATTN_OK;
}

// Whether a handle of this dtype runs on the fp32 SIMT kernels.
bool uses_simt(int dtype) { return dtype == TRI_ATTN_F32; }

size_t base_bytes(int B, int N, int D, int h, int dtype) {
  const size_t es = tri_elem_size(dtype);                              // weights, intermediates
  const size_t cells = (size_t)B * N * N;
  size_t bytes = 0;
  bytes += (size_t)(4 * D + h + 16) * D * es + (size_t)D * D * es;   // packed weights
  bytes += (size_t)(5 * D + h) * sizeof(float);                       // gamma beta bg bo Wb
  bytes += 5 * cells * D * es;                                         // q k v g o
  bytes += (size_t)B * h * N * N * sizeof(float);                      // bias plane
  return bytes + 256;
}

}  // namespace

size_t tri_elem_size(int dtype) { return dtype == TRI_ATTN_F32 ? 4 : 2; }

extern "C" {

const char* tri_attn_status_string(int status) {
  switch (status) {
    case TRI_ATTN_OK: return "ok";
    case TRI_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case TRI_ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case TRI_ATTN_ERR_CUDA: return "CUDA runtime error";
    case TRI_ATTN_ERR_OOM: return "out of device memory";
    case TRI_ATTN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case TRI_ATTN_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

int tri_attn_workspace_bytes(int B, int N, int D, int h, int dtype, size_t* bytes) {
  if (!bytes) return TRI_ATTN_ERR_INVALID_ARG;
  int st = check_shape(B, N, D, h, dtype);
  if (st) return st;
  *bytes = base_bytes(B, N, D, h, dtype) +
           (uses_simt(dtype) ? 0 : tri_tc_extra_bytes(B, N, D, h));
  return TRI_ATTN_OK;
}

int tri_attn_create(tri_attn_t* out, int B, int N, int D, int h, int dtype, int mode,
                    const void* ln_gamma, const void* ln_beta, const void* Wq, const void* Wk,
                    const void* Wv, const void* Wg, const void* bg, const void* Wb,
                    const void* Wo, const void* bo, void* stream) {
  if (!out) return TRI_ATTN_ERR_INVALID_ARG;
  *out = nullptr;
  int st = check_shape(B, N, D, h, dtype);
  if (st) return st;
  if (!tri_mode_valid(mode)) return TRI_ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {ln_gamma, ln_beta, Wq, Wk, Wv, Wg, bg, Wb, Wo, bo};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return TRI_ATTN_ERR_INVALID_ARG;

  cudaStream_t s = (cudaStream_t)stream;
  tri_attn_s* t = (tri_attn_s*)calloc(1, sizeof(tri_attn_s));
  if (!t) return TRI_ATTN_ERR_OOM;
  t->B = B; t->N = N; t->D = D; t->h = h; t->d = D / h;
  t->dtype = dtype; t->mask_mode = tri_mask_mode(mode); t->ending = tri_ending(mode);
  t->cells = (long long)B * N * N;
  t->wait_limit = TRI_DEFAULT_WAIT_LIMIT;
  t->simt = uses_simt(dtype);
  cudaError_t e = cudaGetDevice(&t->device);

  const size_t es = tri_elem_size(dtype);
  const size_t act = (size_t)t->cells * D * es;
  const size_t nproj_pad = (size_t)4 * D + h + 16;
  auto alloc = [&](void** p, size_t n) {
    if (e == cudaSuccess) e = cudaMalloc(p, n);
    if (e == cudaSuccess) t->bytes_owned += n;
  };
  alloc(&t->w_proj, nproj_pad * D * es);
  alloc(&t->w_out, (size_t)D * D * es);
  alloc((void**)&t->gamma, D * sizeof(float));
  alloc((void**)&t->beta, D * sizeof(float));
  alloc((void**)&t->bg, D * sizeof(float));
  alloc((void**)&t->bo, D * sizeof(float));
  alloc((void**)&t->wb_f32, (size_t)h * D * sizeof(float));
  alloc(&t->q, act); alloc(&t->k, act); alloc(&t->v, act); alloc(&t->g, act); alloc(&t->o, act);
  alloc((void**)&t->bias, (size_t)B * h * N * N * sizeof(float));
  alloc((void**)&t->dev_err, 256);
  if (e == cudaSuccess) e = cudaMemsetAsync(t->dev_err, 0, 256, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(t->w_proj, 0, nproj_pad * D * es, s);
  if (e == cudaSuccess) e = to_f32(ln_gamma, dtype, D, t->gamma, s);
  if (e == cudaSuccess) e = to_f32(ln_beta, dtype, D, t->beta, s);
  if (e == cudaSuccess) e = to_f32(bg, dtype, D, t->bg, s);
  if (e == cudaSuccess) e = to_f32(bo, dtype, D, t->bo, s);
  if (e == cudaSuccess) e = to_f32(Wb, dtype, h * D, t->wb_f32, s);
  if (e == cudaSuccess) {
    if (dtype == TRI_ATTN_F32) {
      e = tri_f32_pack_weights(t, Wq, Wk, Wv, Wg, Wb, Wo, s);
    } else {
      e = tri_tc_init(t, Wq, Wk, Wv, Wg, Wb, Wo, s);
    }
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    free_all(t);
    return cuda_status(e);
  }
  *out = t;
  return TRI_ATTN_OK;
}

int tri_attn_forward(tri_attn_t t, void* stream, const void* pair_repr, const int32_t* pair_mask,
                     void* out) {
  if (!t || !pair_repr || !pair_mask || !out) return TRI_ATTN_ERR_INVALID_ARG;
  if (!aligned16(pair_repr) || !aligned16(out) || ((uintptr_t)pair_mask & 3u))
    return TRI_ATTN_ERR_INVALID_ARG;
  const size_t xbytes = (size_t)t->cells * t->D * tri_elem_size(t->dtype);
  const char* xo = (const char*)out;
  const char* xi = (const char*)pair_repr;
  if (xo < xi + xbytes && xi < xo + xbytes) return TRI_ATTN_ERR_INVALID_ARG;
  const char* mi = (const char*)pair_mask;
  const size_t mbytes = (size_t)t->cells * sizeof(int32_t);
  if (xo < mi + mbytes && mi < xo + xbytes) return TRI_ATTN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (t->dtype == TRI_ATTN_F32) {
    e = tri_f32_forward(t, s, (const float*)pair_repr, pair_mask, (float*)out);
  } else {
    e = tri_tc_forward(t, s, pair_repr, pair_mask, out);
  }
  return cuda_status(e);
}

int tri_attn_sync_check(tri_attn_t t, void* stream) {
  if (!t) return TRI_ATTN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  unsigned int err = 0;
  e = cudaMemcpy(&err, t->dev_err, sizeof(err), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  if (err) {
    e = cudaMemset(t->dev_err, 0, sizeof(err));
    if (e != cudaSuccess) return cuda_status(e);
    return (err & TRI_DEV_ERR_TIMEOUT) ? TRI_ATTN_ERR_DEVICE_TIMEOUT : TRI_ATTN_ERR_DEVICE_CHECK;
  }
  return TRI_ATTN_OK;
}

int tri_attn_forward_host(tri_attn_t t, void* stream, const void* pair_repr_host,
                          const int32_t* pair_mask_host, void* out_host) {
  if (!t || !pair_repr_host || !pair_mask_host || !out_host) return TRI_ATTN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t xbytes = (size_t)t->cells * t->D * tri_elem_size(t->dtype);
  const size_t mbytes = (size_t)t->cells * sizeof(int32_t);
  cudaError_t e = cudaSuccess;
  if (!t->stage_x) {
    e = cudaMalloc(&t->stage_x, xbytes);
    if (e == cudaSuccess) e = cudaMalloc((void**)&t->stage_mask, mbytes);
    if (e == cudaSuccess) e = cudaMalloc(&t->stage_out, xbytes);
    if (e != cudaSuccess) return cuda_status(e);
    t->bytes_owned += 2 * xbytes + mbytes;
  }
  if (t->dtype == TRI_ATTN_BF16 && !t->timing) {
    // Copies overlapped with the kernels (chunked).
    e = tri_tc_forward_host(t, s, pair_repr_host, pair_mask_host, out_host, t->stage_x,
                            t->stage_mask, t->stage_out);
    if (e != cudaSuccess) return cuda_status(e);
    return tri_attn_sync_check(t, stream);
  }
  e = cudaMemcpyAsync(t->stage_x, pair_repr_host, xbytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(t->stage_mask, pair_mask_host, mbytes, cudaMemcpyHostToDevice, s);
  int st = e == cudaSuccess ? tri_attn_forward(t, stream, t->stage_x, t->stage_mask, t->stage_out)
                            : cuda_status(e);
  if (st == TRI_ATTN_OK) {
    e = cudaMemcpyAsync(out_host, t->stage_out, xbytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) st = cuda_status(e);
  }
  if (st != TRI_ATTN_OK) {
    // Copies already queued may still touch the caller's host buffers.
    cudaStreamSynchronize(s);
    return st;
  }
  return tri_attn_sync_check(t, stream);
}

int tri_attn_destroy(tri_attn_t t) {
  free_all(t);
  return TRI_ATTN_OK;
}

int tri_attn_enable_kernel_timing(tri_attn_t t, int enable) {
  if (!t) return TRI_ATTN_ERR_INVALID_ARG;
  if (enable && !t->timing) {
    for (int i = 0; i < 8; ++i) {
      cudaError_t e = cudaEventCreate(&t->marks[i]);
      if (e != cudaSuccess) {
        for (int k = 0; k < i; ++k) cudaEventDestroy(t->marks[k]);
        return cuda_status(e);
      }
    }
    t->timing = 1;
    t->n_marks = 0;
  } else if (!enable && t->timing) {
    for (int i = 0; i < 8; ++i) cudaEventDestroy(t->marks[i]);
    t->timing = 0;
    t->n_marks = 0;
  }
  return TRI_ATTN_OK;
}

int tri_attn_kernel_times(tri_attn_t t, float* ms, const char** names, int* n) {
  if (!t || !ms || !n || *n < 0) return TRI_ATTN_ERR_INVALID_ARG;
  if (!t->timing || t->n_marks < 2) {
    *n = 0;
    return TRI_ATTN_OK;
  }
  const int k = t->n_marks - 1;
  if (*n < k) return TRI_ATTN_ERR_INVALID_ARG;
  cudaError_t e = cudaEventSynchronize(t->marks[k]);
  for (int i = 0; i < k && e == cudaSuccess; ++i) {
    e = cudaEventElapsedTime(&ms[i], t->marks[i], t->marks[i + 1]);
    if (names) names[i] = t->mark_names[i + 1];
  }
  if (e != cudaSuccess) return cuda_status(e);
  *n = k;
  return TRI_ATTN_OK;
}

void* tri_attn_debug_tensor(tri_attn_t t, const char* name, int64_t* row_stride) {
  if (!t || !name) return nullptr;
  int64_t ld = t->D;
  void* p = nullptr;
  if (!strcmp(name, "q")) p = t->q;
  else if (!strcmp(name, "k")) p = t->k;
  else if (!strcmp(name, "v")) p = t->v;
  else if (!strcmp(name, "g")) p = t->g;
  else if (!strcmp(name, "o")) p = t->o;
  else if (!strcmp(name, "bias")) {
    p = t->bias;
    ld = t->simt ? t->N : tri_tc_bias_row_stride(t);
  }
  if (p && row_stride) *row_stride = ld;
  return p;
}

int tri_attn_kernel_path(tri_attn_t t) {
  if (!t) return -TRI_ATTN_ERR_INVALID_ARG;
  return t->simt ? TRI_ATTN_PATH_SIMT : TRI_ATTN_PATH_TENSOR_CORE;
}

int tri_attn_set_wait_limit(tri_attn_t t, long long spins) {
  if (!t || spins < 0) return TRI_ATTN_ERR_INVALID_ARG;
  t->wait_limit = spins ? spins : TRI_DEFAULT_WAIT_LIMIT;
  return TRI_ATTN_OK;
}

}  // extern "C"
