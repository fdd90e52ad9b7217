// Host side of the bf16 tensor-core path of triangular self-attention,
// starting and ending node (sm_103a): tensor maps, launchers, the
// device-buffer forward and the host-buffer pipeline that overlaps the host
// copies with chunks of the same kernels.
//
// The kernels live in their own translation units:
//
//   tc_k1.cu  ln_proj_tc   LayerNorm + the concatenated q|k|v|g projection
//                          (tcgen05, TMEM accumulators); the h pair-bias outputs
//                          from the LayerNorm's statistics pass
//   tc_k2.cu  bias_rows    the attention's fp16 bias plane, rows minus their max
//             mask_summary(_cols)  keep bits of every line
//             row_attn_tc  flash-style line attention (S and O in TMEM)
//   tc_k3.cu  gate_out_tc  g * o as the A operand of the output projection
//
// Every shape with D in {32, 64, 128} and d = D / h in {16, 32, 64} has its
// instantiation; the launchers pick it.
//
// Passages followed: POPCORNBENCH "Kimi-K2.6 l2_p6", forward op list steps
// 1-18 and layer definitions; "FW-GLM-5-1 l2_p6", quoted Model.forward.
#include <math.h>
#include <stddef.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "tc_kernels.cuh"

using namespace tri_tc;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  }
  return fn;
}

// Tiled map over a row-major tensor of `rank` dims (dims[0] innermost).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
              const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
              CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, dt, rank, const_cast<void*>(base), dims, strides_bytes, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA swizzle of rows `bytes` long (32, 64 or 128): the tile layout the
// kernels' shared-memory descriptors name.
CUtensorMapSwizzle swizzle_for(int bytes) {
  return bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                      : bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}

// Rows of D bf16 channels (row-major, `rows` of them), loaded one channel
// half (up to 64 channels, swizzled over its own length) x box_rows rows at a
// time.
bool map_rows_bf16(CUtensorMap* m, const void* base, long long rows, int D, int box_rows) {
  const int half_bytes = D >= 64 ? 128 : 2 * D;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {(cuuint32_t)half_bytes / 2, (cuuint32_t)box_rows};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                  swizzle_for(half_bytes));
}

// A (B, N, N, D) bf16 activation seen as (channel, position x along a line,
// line a, batch b): lines are the grid's rows (starting node: cell (a, x)) or
// its columns (ending node: cell (x, a)). Box: one head (d channels, rows of
// 2d bytes swizzled over their length) x box_x positions of one line.
bool map_lines(CUtensorMap* m, const void* base, int B, int N, int D, int d, int box_x,
               bool ending,
               CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t cell = (cuuint64_t)D * 2, row = (cuuint64_t)N * cell;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {ending ? row : cell, ending ? cell : row, (cuuint64_t)N * row};
  cuuint32_t box[4] = {(cuuint32_t)d, (cuuint32_t)box_x, 1, 1};
  return make_map(m, dt, 4, base, dims, strides, box, swizzle_for(2 * d));
}

// K3's view of a (B, N, N, D) bf16 activation as (channel, x, y, z): in cell
// order (x = cell, y = z = 0) or by columns (x = grid row i, y = column j,
// z = batch b). Box: box_ch channels x box_x positions along x.
bool map_k3(CUtensorMap* m, const void* base, const tri_attn_s* t, bool cols, int box_ch,
            int box_x, CUtensorMapSwizzle swz) {
  const cuuint64_t D = (cuuint64_t)t->D;
  const cuuint64_t cell = D * 2, row = (cuuint64_t)t->N * cell, cells = (cuuint64_t)t->cells;
  const cuuint64_t dims_flat[4] = {D, cells, 1, 1}, strides_flat[3] = {cell, cell * cells,
                                                                       cell * cells};
  const cuuint64_t dims_cols[4] = {D, (cuuint64_t)t->N, (cuuint64_t)t->N, (cuuint64_t)t->B};
  const cuuint64_t strides_cols[3] = {row, cell, row * (cuuint64_t)t->N};
  cuuint32_t box[4] = {(cuuint32_t)box_ch, (cuuint32_t)box_x, 1, 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, cols ? dims_cols : dims_flat,
                  cols ? strides_cols : strides_flat, box, swz);
}

// The host-buffer forward moves x in 4 to kXChunks chunks (about 16 MB each,
// measured best) and K2, K3 and out in up to kHostChunks chunks; its events
// are start, mask copied, one per x chunk copied, one per out chunk formed,
// done.
constexpr int kXChunks = 8;
constexpr int kHostChunks = 12;
constexpr int kHostEvents = 3 + 2 * kHostChunks;

struct TcState {
  k1::Consts consts;         // LayerNorm / gate-bias / pair-bias weights (fp32)
  k1::Maps m1;               // K1 maps (x is set per forward)
  k2::Maps m2;               // K2 maps
  k3::Maps m3;               // K3 maps, cell-order tiles (out is set per forward)
  CUtensorMap map_gc, map_oc;   // K3 loads, column tiles
  int R;                     // K2 lines per work unit
  float v_scale;             // v is stored in fp16 times this power of 2
  float* bias32;             // (B, h, N, N) fp32 pair bias in cell order (K1's output)
  unsigned char* row_any;    // (B*N) mask rows keeping some key
  int* line_tiles;           // (B*N) leading key sub-tiles each mask row needs
  uint32_t* mbits;           // (B*N, words) mask bits
  int words;
  int num_sms;
  int Nb;
  // Host-buffer pipeline (created at its first use): copy streams and events.
  cudaStream_t copy_in, copy_out;
  cudaEvent_t ev[kHostEvents];
};

int round_up(int a, int b) { return (a + b - 1) / b * b; }

// n bf16 values times a power of 2 (exact).
__global__ void scale_bf16(__nv_bfloat16* p, long long n, float s) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = __float2bfloat16_rn(__bfloat162float(p[i]) * s);
}


}  // namespace

bool tri_tc_shape_ok(int D, int h) { return tc_shape_ok(D, h); }

bool tri_tc_supported(int B, int N, int D, int h) {
  const long long cells = (long long)B * N * N;
  return tc_shape_ok(D, h) && N >= 1 && N <= 8192 && cells < (1ll << 31) &&
         (long long)B * N < (1ll << 31) / 8;
}

size_t tri_tc_extra_bytes(int B, int N, int, int h) {
  // the attention's fp16 bias plane (rows padded to Nb) beside K1's fp32 one;
  // plus the mask summary
  const size_t Nb = (size_t)round_up(N, 8);
  return (size_t)B * h * N * Nb * 2 + (size_t)B * N * 5 + (size_t)B * N * 2 * ((N + 63) / 64) * 4 +
         1024;
}

cudaError_t tri_tc_init(tri_attn_s* t, const void* Wq, const void* Wk, const void* Wv,
                        const void* Wg, const void*, const void* Wo, cudaStream_t s) {
  TcState* st = (TcState*)calloc(1, sizeof(TcState));
  if (!st) return cudaErrorMemoryAllocation;
  t->tc = st;
  const int B = t->B, N = t->N, D = t->D, h = t->h;
  st->Nb = round_up(N, 8);
  cudaError_t e = cudaDeviceGetAttribute(&st->num_sms, cudaDevAttrMultiProcessorCount, t->device);
  // K1 writes the fp32 plane the handle allocated (cell order); the attention
  // reads an fp16 plane with rows padded to Nb (TMA strides are multiples of 16
  // bytes), which takes the handle's bias pointer.
  if (e == cudaSuccess) {
    st->bias32 = t->bias;
    t->bias = nullptr;
    e = cudaMalloc((void**)&t->bias, (size_t)B * h * N * st->Nb * 2);
  }
  st->words = 2 * ((N + k2::BK - 1) / k2::BK);   // two 32-key words per 64-key tile
  st->R = k2_lines_per_unit(t->d);
  if (e == cudaSuccess) e = cudaMalloc((void**)&st->row_any, (size_t)B * N);
  if (e == cudaSuccess) e = cudaMalloc((void**)&st->line_tiles, (size_t)B * N * 4);
  if (e == cudaSuccess) e = cudaMalloc((void**)&st->mbits, (size_t)B * N * st->words * 4);
  const size_t wbytes = (size_t)D * D * 2;
  const void* mats[4] = {Wq, Wk, Wv, Wg};
  for (int m = 0; m < 4 && e == cudaSuccess; ++m)
    e = cudaMemcpyAsync((char*)t->w_proj + m * wbytes, mats[m], wbytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(t->w_out, Wo, wbytes, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return e;
  // fp32 copies of the small parameters, made by tri_attn_create, go by value.
  memset(&st->consts, 0, sizeof(st->consts));
  if (e == cudaSuccess) e = cudaMemcpyAsync(st->consts.gamma, t->gamma, D * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st->consts.beta, t->beta, D * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st->consts.bg, t->bg, D * 4, cudaMemcpyDeviceToHost, s);
  // Wb arrives as [h][D]; consts.gw holds its rows kMaxD apart.
  float wb[kMaxH * kMaxD];
  if (e == cudaSuccess) e = cudaMemcpyAsync(wb, t->wb_f32, (size_t)h * D * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  for (int hd = 0; hd < h; ++hd) memcpy(st->consts.gw[hd], wb + (size_t)hd * D, (size_t)D * 4);
  // Fold gamma and beta into the bias projection (see k1::Consts).
  for (int hd = 0; hd < h; ++hd) {
    double gs = 0.0, bs = 0.0;
    for (int c = 0; c < D; ++c) {
      const double wbv = st->consts.gw[hd][c];
      bs += (double)st->consts.beta[c] * wbv;
      st->consts.gw[hd][c] = (float)((double)st->consts.gamma[c] * wbv);
      gs += st->consts.gw[hd][c];
    }
    st->consts.gws[hd] = (float)gs;
    st->consts.bw[hd] = (float)bs;
  }

  // v = Wv x_hat goes to fp16. Every LayerNorm output obeys |x_hat_c| <=
  // |gamma_c| sqrt(D - 1) + |beta_c| (no entry of D values lies more than
  // sqrt(D - 1) standard deviations from their mean), so |v_e| <= sum_c
  // |Wv[e][c]| (|gamma_c| sqrt(D - 1) + |beta_c|) for any input; v is stored
  // times the power of 2 that keeps this bound (with a margin for the bf16
  // rounding of x_hat) below 2^15.
  {
    static_assert(sizeof(__nv_bfloat16) == 2, "bf16 weights");
    uint16_t* wv = (uint16_t*)malloc((size_t)D * D * 2);
    if (!wv) return cudaErrorMemoryAllocation;
    e = cudaMemcpy(wv, Wv, (size_t)D * D * 2, cudaMemcpyDeviceToHost);
    double bound = 0.0;
    const double sq = sqrt((double)(D - 1));
    for (int r = 0; r < D && e == cudaSuccess; ++r) {
      double acc = 0.0;
      for (int c = 0; c < D; ++c) {
        uint32_t bits = (uint32_t)wv[(size_t)r * D + c] << 16;
        float w;
        memcpy(&w, &bits, 4);
        acc += fabs((double)w) * (fabs((double)st->consts.gamma[c]) * sq + fabs((double)st->consts.beta[c]));
      }
      bound = std::max(bound, acc);
    }
    free(wv);
    if (e != cudaSuccess) return e;
    bound *= 1.02;
    st->v_scale = 1.0f;
    while (bound * st->v_scale >= 32768.0 && st->v_scale > 0x1p-100f) st->v_scale *= 0.5f;
    // The scale goes into the packed Wv rows (rows 2D .. 3D - 1 of [Wq;Wk;Wv;Wg]):
    // a power of 2, so the bf16 weights scale exactly.
    if (st->v_scale != 1.0f) {
      const long long n = (long long)D * D;
      scale_bf16<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
          (__nv_bfloat16*)t->w_proj + 2ll * D * D, n, st->v_scale);
      e = cudaGetLastError();
      if (e == cudaSuccess) e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return e;
    }
  }

  const long long cells = t->cells;
  const int d = t->d, half_bytes = D >= 64 ? 128 : 2 * D, kvk = k2_keys_per_stage(d);
  bool ok = map_rows_bf16(&st->m1.w, t->w_proj, 4 * D, D, 2 * D);
  ok = ok && map_lines(&st->m2.q, t->q, B, N, D, d, k2::BQ, t->ending);
  ok = ok && map_lines(&st->m2.k, t->k, B, N, D, d, kvk, t->ending);
  ok = ok && map_lines(&st->m2.v, t->v, B, N, D, d, kvk, t->ending, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  ok = ok && map_lines(&st->m2.o, t->o, B, N, D, d, 32, t->ending);
  {
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)B * h};
    cuuint64_t strides[2] = {(cuuint64_t)st->Nb * 2, (cuuint64_t)N * st->Nb * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)k2::BQ, 1};   // 128-byte rows for SWIZZLE_128B
    ok = ok && make_map(&st->m2.b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, t->bias, dims, strides,
                        box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const CUtensorMapSwizzle hsw = swizzle_for(half_bytes);
  ok = ok && map_k3(&st->m3.g, t->g, t, false, half_bytes / 2, 128, hsw);
  ok = ok && map_k3(&st->map_gc, t->g, t, true, half_bytes / 2, 128, hsw);
  {
    void* outs[4] = {t->q, t->k, t->v, t->g};
    CUtensorMap* maps[4] = {&st->m1.q, &st->m1.k, &st->m1.v, &st->m1.g};
    for (int m = 0; m < 4 && ok; ++m) {
      cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)cells};
      cuuint64_t strides[1] = {(cuuint64_t)D * 2};
      cuuint32_t box[2] = {32, 32};
      // v is fp16 (the attention's P V operand), q, k and g bf16.
      ok = make_map(maps[m], m == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    2, outs[m], dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    }
  }
  ok = ok && map_k3(&st->m3.o, t->o, t, false, half_bytes / 2, 128, hsw);
  ok = ok && map_k3(&st->map_oc, t->o, t, true, half_bytes / 2, 128, hsw);
  ok = ok && map_rows_bf16(&st->m3.wo, t->w_out, D, D, D);
  if (!ok) return cudaErrorInvalidValue;
  e = k1_init();
  if (e == cudaSuccess) e = k2_init();
  if (e == cudaSuccess) e = k3_init();
  return e;
}

int tri_tc_bias_row_stride(const tri_attn_s* t) {
  const TcState* st = (const TcState*)t->tc;
  return st ? st->Nb : t->N;
}

void tri_tc_release(tri_attn_s* t) {
  TcState* st = (TcState*)t->tc;
  if (!st) return;
  if (st->bias32) cudaFree(st->bias32);
  if (st->row_any) cudaFree(st->row_any);
  if (st->line_tiles) cudaFree(st->line_tiles);
  if (st->mbits) cudaFree(st->mbits);
  if (st->copy_in) cudaStreamDestroy(st->copy_in);
  if (st->copy_out) cudaStreamDestroy(st->copy_out);
  for (int i = 0; i < kHostEvents; ++i)
    if (st->ev[i]) cudaEventDestroy(st->ev[i]);
  free(st);
  t->tc = nullptr;
}

namespace {

int num_tiles(const tri_attn_s* t) { return (int)((t->cells + 127) / 128); }

// K1 over tiles tile0 .. tile0 + n - 1 of the grid's cells.
cudaError_t launch_k1(tri_attn_s* t, cudaStream_t s, const CUtensorMap& map_x,
                      const int32_t* mask, int tile0, int n) {
  TcState* st = (TcState*)t->tc;
  k1::Params p1;
  p1.cells = t->cells; p1.N = t->N; p1.h = t->h; p1.mask_mode = t->mask_mode;
  p1.ntiles = n; p1.tile0 = tile0;
  p1.mask = mask;
  p1.bias32 = st->bias32; p1.dev_err = t->dev_err;
  p1.polls = t->wait_limit;
  p1.q_scale = kLog2e / sqrtf((float)t->d);
  const int grid = n < st->num_sms ? n : st->num_sms;
  k1::Maps m = st->m1;
  m.x = map_x;
  return k1_launch(t->D, t->h, grid, s, !t->timing, m, p1, st->consts);
}

// The mask summary of every line.
cudaError_t launch_mask(tri_attn_s* t, cudaStream_t s, const int32_t* mask, int& mark) {
  TcState* st = (TcState*)t->tc;
  const cudaError_t e =
      k2_mask_summary(mask, t->B, t->N, t->ending, st->words, st->mbits, st->row_any, st->line_tiles, s,
                      !t->timing);
  tri_mark(t, s, mark++, t->ending ? "mask_summary_cols" : "mask_summary");
  return e;
}

// The attention's bias plane from K1's (after every K1 tile).
cudaError_t launch_bias_rows(tri_attn_s* t, cudaStream_t s, int& mark) {
  TcState* st = (TcState*)t->tc;
  const cudaError_t e =
      k2_bias_rows(st->bias32, t->B, t->h, t->N, st->Nb, t->ending, (__half*)t->bias, s, !t->timing);
  tri_mark(t, s, mark++, "bias_rows");
  return e;
}

// K2's work units are (b, row group, head, query tile), query tile fastest.
int k2_row_groups(const tri_attn_s* t) {
  const int R = ((const TcState*)t->tc)->R;
  return (t->N + R - 1) / R;
}
int k2_units_per_group(const tri_attn_s* t) { return t->h * ((t->N + k2::BQ - 1) / k2::BQ); }

// K2 over units u0 .. u0 + nu - 1 (any range; the units of one (b, row group)
// pair are consecutive).
cudaError_t launch_k2(tri_attn_s* t, cudaStream_t s, int u0, int nu) {
  TcState* st = (TcState*)t->tc;
  const int N = t->N, h = t->h;
  k2::Params p2;
  p2.B = t->B; p2.N = N; p2.h = h; p2.mask_mode = t->mask_mode;
  p2.row_groups = k2_row_groups(t);
  p2.jtiles = (N + k2::BQ - 1) / k2::BQ;
  p2.unit0 = u0;
  p2.units = nu;
  p2.words = st->words;
  p2.mbits = st->mbits; p2.row_any = st->row_any; p2.line_tiles = st->line_tiles;
  p2.dev_err = t->dev_err;
  p2.polls = t->wait_limit;
  p2.q = (const __nv_bfloat16*)t->q;
  p2.k = (const __nv_bfloat16*)t->k;
  p2.v = (const __half*)t->v;
  p2.v_unscale = 1.0f / st->v_scale;
  p2.sb = (long long)N * N * t->D;
  p2.sl = t->ending ? (long long)t->D : (long long)N * t->D;     // line a: row (starting) or column
  p2.sx = t->ending ? (long long)N * t->D : (long long)t->D;     // position along the line
  p2.bias32 = st->bias32;
  p2.ending = t->ending ? 1 : 0;
  const unsigned g2 = (unsigned)(p2.units < st->num_sms ? p2.units : st->num_sms);
  {
    const int g1 = (int)g2 / p2.jtiles, gq = g1 / h;
    p2.step.jt = (int)g2 % p2.jtiles;
    p2.step.t = g1 % h;
    p2.step.rg = gq % p2.row_groups;
    p2.step.b = gq / p2.row_groups;
  }
  return k2_launch(t->d, (int)g2, s, !t->timing, st->m2, p2);
}

// Store map of K3's bf16 output (cell order or by columns): 32 x 32 boxes.
bool map_out_k3(CUtensorMap* m, void* out, const tri_attn_s* t, bool cols) {
  return map_k3(m, out, t, cols, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// K3's tiles per grid column in column order.
int k3_tiles_per_col(const tri_attn_s* t) { return (t->N + k3::BM - 1) / k3::BM; }

// K3 over tiles tile0 .. tile0 + n - 1, in cell order or in column order
// (map_out made with the same order).
cudaError_t launch_k3(tri_attn_s* t, cudaStream_t s, const CUtensorMap& map_out, int tile0,
                      int n, bool cols) {
  TcState* st = (TcState*)t->tc;
  k3::Params p3;
  p3.cells = t->cells; p3.ntiles = n; p3.tile0 = tile0; p3.bo = t->bo;
  p3.cols = cols ? 1 : 0; p3.N = t->N; p3.tpl = k3_tiles_per_col(t);
  p3.dev_err = t->dev_err; p3.polls = t->wait_limit;
  const int grid = n < st->num_sms ? n : st->num_sms;
  k3::Maps m = st->m3;
  if (cols) {
    m.g = st->map_gc;
    m.o = st->map_oc;
  }
  m.out = map_out;
  return k3_launch(t->D, grid, s, !t->timing, m, p3);
}

}  // namespace

cudaError_t tri_tc_forward(tri_attn_s* t, cudaStream_t s, const void* x, const int32_t* mask,
                           void* out) {
  const int ntiles = num_tiles(t);
  CUtensorMap map_x, map_out;
  if (!map_rows_bf16(&map_x, x, t->cells, t->D, 128) || !map_out_k3(&map_out, out, t, false))
    return cudaErrorInvalidValue;
  int mark = 0;
  tri_mark(t, s, mark++, nullptr);
  cudaError_t e = launch_k1(t, s, map_x, mask, 0, ntiles);
  tri_mark(t, s, mark++, "ln_proj_tc");
  if (e == cudaSuccess) e = launch_mask(t, s, mask, mark);
  if (e == cudaSuccess) e = launch_bias_rows(t, s, mark);
  if (e == cudaSuccess) e = launch_k2(t, s, 0, t->B * k2_row_groups(t) * k2_units_per_group(t));
  tri_mark(t, s, mark++, "row_attn_tc");
  if (e == cudaSuccess) e = launch_k3(t, s, map_out, 0, ntiles, false);
  tri_mark(t, s, mark++, "gate_out_tc");
  return e;
}

// Host buffers in and out, pipelined. x arrives in chunks on a copy stream
// while K1 works on the chunks already on the device (the mask summary runs
// first, during the first copy). Every line's attention needs the whole bias
// plane, so K2 starts after the last K1 chunk; it then runs in chunks of line
// groups, and after each chunk K3 forms the out tiles of the finished lines,
// which are copied back while the next chunk runs: grid rows for the starting
// node, grid columns (a strided copy per batch) for the ending node. dx, dmask,
// dout are the handle's device staging buffers.
cudaError_t tri_tc_forward_host(tri_attn_s* t, cudaStream_t s, const void* xh,
                                const int32_t* maskh, void* outh, void* dx, int32_t* dmask,
                                void* dout) {
  TcState* st = (TcState*)t->tc;
  cudaError_t e = cudaSuccess;
  if (!st->copy_in) {
    e = cudaStreamCreateWithFlags(&st->copy_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st->copy_out, cudaStreamNonBlocking);
    for (int i = 0; i < kHostEvents && e == cudaSuccess; ++i)
      e = cudaEventCreateWithFlags(&st->ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  const bool cols = t->ending;
  const int ntiles = num_tiles(t);
  const size_t row_bytes = (size_t)t->D * 2;
  const long long want = std::min<long long>(
      kXChunks, std::max<long long>(4, (long long)(t->cells * row_bytes >> 24)));
  const int nch = (int)std::min<long long>(ntiles, want);
  const int per = (ntiles + nch - 1) / nch;
  CUtensorMap map_x, map_out;
  if (!map_rows_bf16(&map_x, dx, t->cells, t->D, 128) || !map_out_k3(&map_out, dout, t, cols))
    return cudaErrorInvalidValue;
  cudaEvent_t* ev = st->ev;          // [0] start, [1] mask in, [2 ..] x chunks in, out chunks done
  cudaEvent_t* ev_x = ev + 2;
  cudaEvent_t* ev_o = ev + 2 + kHostChunks;
  cudaEvent_t ev_done = ev[2 + 2 * kHostChunks];
  // The copies start after the work already queued on s.
  e = cudaEventRecord(ev[0], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st->copy_in, ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st->copy_out, ev[0], 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dmask, maskh, (size_t)t->cells * sizeof(int32_t), cudaMemcpyHostToDevice,
                        st->copy_in);
  if (e == cudaSuccess) e = cudaEventRecord(ev[1], st->copy_in);
  for (int i = 0; i < nch && e == cudaSuccess; ++i) {
    const long long c0 = (long long)i * per * 128;
    const long long c1 = std::min((long long)(i + 1) * per * 128, t->cells);
    if (c0 >= c1) break;
    e = cudaMemcpyAsync((char*)dx + c0 * row_bytes, (const char*)xh + c0 * row_bytes,
                        (size_t)(c1 - c0) * row_bytes, cudaMemcpyHostToDevice, st->copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_x[i], st->copy_in);
  }
  int mark = 0;
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev[1], 0);
  if (e == cudaSuccess) e = launch_mask(t, s, dmask, mark);
  for (int i = 0; i < nch && e == cudaSuccess; ++i) {
    const int t0 = i * per, n = std::min(per, ntiles - t0);
    if (n <= 0) break;
    e = cudaStreamWaitEvent(s, ev_x[i], 0);
    if (e == cudaSuccess) e = launch_k1(t, s, map_x, dmask, t0, n);
  }
  if (e == cudaSuccess) e = launch_bias_rows(t, s, mark);
  // K2 chunk boundaries in work units: up to eight equal chunks of whole
  // waves of CTAs (a partial wave takes as long as a full one), the last
  // taking what is left. Each chunk adds a K2 ramp and a K3 launch (~20 us at
  // N = 768) to the K2 -> K3 chain on s, which runs about as fast as the copy
  // back, so a short first chunk gains nothing (a timeline of one-wave-first
  // chunks growing 1.3 times showed the copy stream waiting on that chain). A
  // chunk finishes the lines of the row groups whose units it completes.
  const int groups = t->B * k2_row_groups(t);
  const int upg = k2_units_per_group(t);
  const int units = groups * upg;
  const int wave = st->num_sms;
  const int chunk = wave * std::max(1, (units + 8 * wave - 1) / (8 * wave));
  const int nk2 = (units + chunk - 1) / chunk;
  // Lines (b, a), counted as b * N + a, that the groups before group g cover.
  const int rgs = k2_row_groups(t);
  auto lines_before = [&](int g) -> long long {
    if (g >= groups) return (long long)t->B * t->N;
    return (long long)(g / rgs) * t->N + std::min((g % rgs) * st->R, t->N);
  };
  const long long NN = (long long)t->N * t->N;
  const int tpl = k3_tiles_per_col(t);
  long long lines_done = 0;
  int tile_done = 0;
  for (int i = 0; i < nk2 && e == cudaSuccess; ++i) {
    const int u0 = i * chunk, u1 = std::min(units, u0 + chunk);
    e = launch_k2(t, s, u0, u1 - u0);
    const long long lend = lines_before(u1 / upg);
    if (e != cudaSuccess || lend <= lines_done) continue;
    if (cols) {
      // Column tiles of the finished columns, then one strided copy per batch.
      e = launch_k3(t, s, map_out, (int)(lines_done * tpl), (int)((lend - lines_done) * tpl), true);
      if (e == cudaSuccess) e = cudaEventRecord(ev_o[i], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st->copy_out, ev_o[i], 0);
      const size_t pitch = (size_t)t->N * row_bytes;
      for (long long b = lines_done / t->N; b * t->N < lend && e == cudaSuccess; ++b) {
        const long long j0 = std::max(lines_done - b * t->N, 0LL);
        const long long j1 = std::min(lend - b * t->N, (long long)t->N);
        const size_t off = (size_t)(b * NN + j0) * row_bytes;
        e = cudaMemcpy2DAsync((char*)outh + off, pitch, (const char*)dout + off, pitch,
                              (size_t)(j1 - j0) * row_bytes, (size_t)t->N,
                              cudaMemcpyDeviceToHost, st->copy_out);
      }
      lines_done = lend;
    } else {
      // Cell-order tiles whose grid rows are all finished (the last chunk
      // takes the rest), then one contiguous copy.
      const int tile_end = lend == (long long)t->B * t->N
                               ? ntiles : (int)(std::min(lend * t->N, t->cells) / 128);
      lines_done = lend;
      if (tile_end <= tile_done) continue;
      e = launch_k3(t, s, map_out, tile_done, tile_end - tile_done, false);
      if (e == cudaSuccess) e = cudaEventRecord(ev_o[i], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st->copy_out, ev_o[i], 0);
      const long long c0 = (long long)tile_done * 128;
      const long long c1 = std::min((long long)tile_end * 128, t->cells);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync((char*)outh + c0 * row_bytes, (const char*)dout + c0 * row_bytes,
                            (size_t)(c1 - c0) * row_bytes, cudaMemcpyDeviceToHost, st->copy_out);
      tile_done = tile_end;
    }
  }
  // s finishes only once the last chunk of out is on the host.
  if (e == cudaSuccess) e = cudaEventRecord(ev_done, st->copy_out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_done, 0);
  if (e != cudaSuccess) {
    // Copies already queued may still read or write the caller's host buffers:
    // let them finish before the error reaches the caller.
    cudaStreamSynchronize(st->copy_in);
    cudaStreamSynchronize(st->copy_out);
    cudaStreamSynchronize(s);
  }
  return e;
}
