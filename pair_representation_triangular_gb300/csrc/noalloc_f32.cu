// tri_attn_forward_noalloc: the fp32 forward pass for callers that cannot
// allocate device memory.
//
// Some callers have no way to call cudaMalloc at the point where they need a
// forward pass: code running under a custom allocator or a memory pool that
// forbids outside allocations, plugins handed only input and output buffers by
// their host framework, or real-time loops where an allocation (and the device
// synchronisation it can imply) is not allowed. tri_attn_create allocates its
// weights and workspace, so those callers cannot use it. This entry point takes
// every weight, input and output as a caller pointer and keeps all intermediates
// (packed weights, q, k, v, g, o and the bias plane) in one fixed, file-scope
// device array, so it allocates nothing.
#include "common.cuh"

namespace {

// Fixed scratch of the no-allocation entry point. Every device the library's
// code is loaded on (lazily, at the first call there) holds this array until
// the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array in the current context. In host code the
// array's name is only a host-side stand-in, so kernels must be given this
// address. It is looked up at every call (cheap once the code is loaded), so a
// context that was reset or re-created never receives a stale address.
cudaError_t scratch_address(unsigned char** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = (unsigned char*)p;
  return cudaSuccess;
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// Scratch bytes one call needs: packed weights (projection rows padded to an
// even count), five (cells x D) intermediates and the bias plane, each
// 256-byte aligned.
size_t scratch_bytes(int B, int N, int D, int h) {
  const size_t cells = (size_t)B * N * N;
  return round256((size_t)((4 * D + h + 1) & ~1) * D * 4) + round256((size_t)D * D * 4) +
         5 * round256(cells * D * 4) + round256((size_t)B * h * N * N * 4);
}

}  // namespace

extern "C" int tri_attn_forward_noalloc(int B, int N, int D, int h, int mode,
                                        const float* ln_gamma, const float* ln_beta,
                                        const float* Wq, const float* Wk, const float* Wv,
                                        const float* Wg, const float* bg, const float* Wb,
                                        const float* Wo, const float* bo, void* stream,
                                        const float* pair_repr, const int32_t* pair_mask,
                                        float* out) {
  if (B < 1 || N < 1 || D < 1 || h < 1 || D % h) return TRI_ATTN_ERR_INVALID_ARG;
  if (!tri_mode_valid(mode)) return TRI_ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {ln_gamma, ln_beta, Wq, Wk, Wv, Wg, bg, Wb, Wo, bo, pair_repr, out};
  for (const void* p : ptrs)
    if (!p || ((uintptr_t)p & 15u)) return TRI_ATTN_ERR_INVALID_ARG;
  if (!pair_mask || ((uintptr_t)pair_mask & 3u)) return TRI_ATTN_ERR_INVALID_ARG;
  if (D > 256 || D / h > 128 || (D & 1)) return TRI_ATTN_ERR_UNSUPPORTED;
  if ((long long)B * N * N * D > (1ll << 40)) return TRI_ATTN_ERR_UNSUPPORTED;
  if (scratch_bytes(B, N, D, h) > kNoAllocScratchBytes)
    return TRI_ATTN_ERR_UNSUPPORTED;      // the problem does not fit the fixed scratch

  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  const size_t cells = (size_t)B * N * N;
  TriF32Raw a;
  a.B = B; a.N = N; a.D = D; a.h = h;
  a.mask_mode = tri_mask_mode(mode); a.ending = tri_ending(mode);
  a.gamma = ln_gamma; a.beta = ln_beta; a.Wq = Wq; a.Wk = Wk; a.Wv = Wv; a.Wg = Wg;
  a.bg = bg; a.Wb = Wb; a.Wo = Wo; a.bo = bo;
  a.x = pair_repr; a.mask = pair_mask; a.out = out;
  // Every byte of the scratch that a kernel reads is written earlier in the same
  // call (weights packed first, then each intermediate in full), so nothing
  // needs clearing between calls.
  unsigned char* p = base;
  a.w_proj = (float*)p; p += round256((size_t)((4 * D + h + 1) & ~1) * D * 4);
  a.w_out = (float*)p;  p += round256((size_t)D * D * 4);
  float** acts[5] = {&a.q, &a.k, &a.v, &a.g, &a.o};
  for (float** ap : acts) { *ap = (float*)p; p += round256(cells * D * 4); }
  a.bias = (float*)p;
  e = tri_f32_forward_raw(a, (cudaStream_t)stream);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}
