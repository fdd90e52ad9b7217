// bf16 tensor-core path (placeholder until the tcgen05 kernels land).
#include "common.cuh"

bool tri_tc_supported(int, int, int, int) { return false; }
size_t tri_tc_extra_bytes(int, int, int, int) { return 0; }
cudaError_t tri_tc_init(tri_attn_s*, const void*, const void*, const void*, const void*,
                        const void*, const void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
void tri_tc_release(tri_attn_s*) {}
cudaError_t tri_tc_forward(tri_attn_s*, cudaStream_t, const void*, const int32_t*, void*) {
  return cudaErrorNotSupported;
}
