// Interface between the host side of the bf16 tensor-core path (kernels_tc.cu)
// and the translation units that hold its kernels (tc_k1.cu, tc_k2.cu,
// tc_k3.cu): the kernel parameter blocks and one launcher per kernel family,
// which picks the instantiation for the handle's shape.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tc_shapes.h"

namespace tri_tc {

namespace k1 {
// LayerNorm and bias parameters travel by value in the kernel parameter block
// (constant bank): every read index is known at compile time.
// gw[t][c] = gamma[c] Wb[t][c], gws[t] = sum_c gw[t][c], bw[t] = sum_c beta[c] Wb[t][c]:
// with t_c = (x_c - mean) rstd, bias[t] = sum_c x_hat_c Wb[t][c]
// = rstd (sum_c (x_c - K) gw[t][c] - (mean - K) gws[t]) + bw[t] for any shift K.
// Entries past D channels or h heads are zero.
struct alignas(16) Consts {     // 16-byte aligned: rows are read as float2 pairs
  float gamma[kMaxD], beta[kMaxD], bg[kMaxD], gw[kMaxH][kMaxD], gws[kMaxH], bw[kMaxH];
};
static_assert(offsetof(Consts, gw) % 16 == 0 && offsetof(Consts, beta) % 16 == 0,
              "parameter rows must stay 8-byte aligned");

struct Params {
  long long cells;
  int N, h, mask_mode, ntiles;       // this launch: tiles tile0 .. tile0 + ntiles - 1
  int tile0;
  const int32_t* mask;
  float* bias32;               // (B, h, N, N) fp32 in cell order, scaled by log2(e)
  unsigned int* dev_err;
  long long polls;
  float q_scale;               // q is stored times log2(e) / sqrt(d)
};

// x: loads (channel, cell), box (channels of one half, 128 cells). w: the
// resident [Wq;Wk;Wv;Wg] (channel, output), box (one half, 2D outputs). q, k,
// v, g: stores (channel, cell), 32 x 32 boxes.
struct Maps {
  CUtensorMap x, w, q, k, v, g;
};
}  // namespace k1

namespace k2 {
// A step of gridDim.x units written in the units' mixed radix (query tile,
// head, row group, batch; query tile fastest).
struct UnitStep {
  int jt, t, rg, b;
};

struct Params {
  int B, N, h, mask_mode, row_groups, jtiles, words;
  int unit0, units;               // this launch: units unit0 .. unit0 + units - 1
  UnitStep step;                  // gridDim.x in unit digits
  const uint32_t* mbits;          // (B*N rows, words): bit k = pair_mask[b, r, k] != 0, k < N
  const unsigned char* row_any;   // (B*N rows): the mask row keeps some key
  // (B*N rows): leading 64-key sub-tiles the row needs: up to its last kept
  // key, or all of them when it keeps none (weight 1 on every real key)
  const int* line_tiles;
  unsigned int* dev_err;
  long long polls;
  // The same q, k, v and bias plane as raw tensors, for the exact recomputation
  // of a query row whose sums left the fp32 range: element (b, line a, position
  // x, channel e) of q, k or v sits at b * sb + a * sl + x * sx + e.
  const __nv_bfloat16 *q, *k;
  const __half* v;                // fp16, times v_scale (a power of 2)
  float v_unscale;                // 1 / v_scale
  long long sb, sl, sx;
  const float* bias32;            // (B, h, N, N) fp32 cell order, log2(e) * bias, -inf where dropped
  int ending;                     // the key k of query a is cell (k, a) instead of (a, k)
};

// q, k, v: loads (channel, position, line, batch), boxes (d, 128 | KVK, 1, 1).
// b: the fp16 bias plane (key, query, b * h + t), box (64, 128, 1). o: stores,
// box (d, 32, 1, 1).
struct Maps {
  CUtensorMap q, k, v, b, o;
};
}  // namespace k2

namespace k3 {
struct Params {
  long long cells;
  int ntiles, tile0;              // this launch: tiles tile0 .. tile0 + ntiles - 1
  // Tile order. cols = 0: tile t is cells t*128 .. t*128 + 127 in memory order
  // (maps (channel, cell, 1, 1)). cols = 1: tile t is rows x .. x + 127 of one
  // column j of the grid of batch b, with tpl tiles per column (maps (channel,
  // i, j, b)), so a run of tiles covers whole columns.
  int cols, N, tpl;
  const float* bo;
  unsigned int* dev_err;
  long long polls;
};

// g, o: loads, box (channels of one half, 128); wo: Wo (channel, output), box
// (one half, D); out: stores, 32 x 32 boxes.
struct Maps {
  CUtensorMap g, o, wo, out;
};
}  // namespace k3

// Launch with the programmatic-stream-serialization attribute: the kernel may
// begin while the previous kernel on the stream finishes (it waits for that
// kernel's completion itself, see pdl_wait). After any other stream operation
// the attribute has no effect and ordering is the stream's usual one.
template <typename... ExpTypes, typename... ActTypes>
cudaError_t launch_pdl(bool pdl, void (*kernel)(ExpTypes...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, ActTypes&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<ActTypes&&>(args)...);
}

// Launchers: each picks the kernel instantiated for the shape and returns the
// launch status; `pdl` requests the programmatic dependent launch (off while
// events are recorded between the kernels). *_init sets the shared-memory size
// of every instantiation.
cudaError_t k1_init();
cudaError_t k1_launch(int D, int h, int grid, cudaStream_t s, bool pdl, const k1::Maps& m,
                      const k1::Params& p, const k1::Consts& c);

cudaError_t k2_init();
int k2_lines_per_unit(int d);
int k2_keys_per_stage(int d);
cudaError_t k2_launch(int d, int grid, cudaStream_t s, bool pdl, const k2::Maps& m,
                      const k2::Params& p);
cudaError_t k2_mask_summary(const int32_t* mask, int B, int N, bool ending, int words,
                            uint32_t* bits, unsigned char* any, int* tiles, cudaStream_t s, bool pdl);
cudaError_t k2_bias_rows(const float* C, int B, int h, int N, int Nb, bool ending, __half* P,
                         cudaStream_t s, bool pdl);

cudaError_t k3_init();
cudaError_t k3_launch(int D, int grid, cudaStream_t s, bool pdl, const k3::Maps& m,
                      const k3::Params& p);

}  // namespace tri_tc
