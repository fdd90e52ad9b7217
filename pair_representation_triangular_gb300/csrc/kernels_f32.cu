// fp32 SIMT path of triangular self-attention (starting and ending node).
//
// Three kernels, in the split of the "Kimi-K2.6 l2_p6" POPCORNBENCH page
// (preprocess / attention / finalize), written for fp32 accuracy rather than
// tensor-core throughput:
//   ln_proj_f32    LayerNorm + the five projections of every cell, gate sigmoid,
//                  pair bias scattered to its (B, h, N, N) plane;
//   row_attn_f32   per (line, head, 128 queries): logits with the shared pair
//                  bias, mask replacement by -1e9, online softmax over keys
//                  staged 32 at a time, P.V. A line is a row i of the grid
//                  (starting node) or a column j (ending node): its cell x
//                  sits at b N^2 + a sa + x sx with (sa, sx) = (N, 1) or (1, N);
//   gate_out_f32   g * o followed by the output projection and its bias.
#include <math.h>

#include "common.cuh"

namespace {

constexpr int kCellsPerBlock = 32;   // cells per block in the two projection kernels
constexpr int kProjThreads = 256;
constexpr int kQueriesPerBlock = 128;
constexpr int kKeyChunk = 32;

// Transpose-pack W (rows x D, nn.Linear layout) into dst[e * ld + col0 + r].
__global__ void pack_transpose_f32(const float* __restrict__ W, int rows, int D,
                                   float* __restrict__ dst, int ld, int col0) {
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * D) return;
  int r = idx / D, e = idx % D;
  dst[(size_t)e * ld + col0 + r] = W[idx];
}

// Shared-memory operand of the two projection kernels: the block's 32 cells
// stored channel-major, xt[e * kXtLd + c], rows padded to 36 floats so that
// four consecutive cells load as one aligned 16-byte vector.
constexpr int kXtLd = kCellsPerBlock + 4;

// Row stride of the packed projection weights [D][4D + h], rounded up to an
// even count so that every output pair loads as one aligned float2.
inline int proj_ld(int D, int h) { return (4 * D + h + 1) & ~1; }

// acc[i][c] += sum_e xt[e][c0 + c] * Wt[e][o0 + i] for i < 2, c < CT: one
// thread's 2-output x CT-cell tile of a skinny GEMM over D channels.
template <int CT>
__device__ __forceinline__ void tile_gemm(const float* __restrict__ xt, int c0, int D,
                                          const float* __restrict__ Wt, int ld, int o0,
                                          float (&acc)[2][CT]) {
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int c = 0; c < CT; ++c) acc[i][c] = 0.f;
#pragma unroll 4
  for (int e = 0; e < D; ++e) {
    const float2 w = *(const float2*)(Wt + (size_t)e * ld + o0);
    float xv[CT];
#pragma unroll
    for (int c = 0; c < CT; c += 4) *(float4*)&xv[c] = *(const float4*)(xt + e * kXtLd + c0 + c);
#pragma unroll
    for (int c = 0; c < CT; ++c) {
      acc[0][c] = fmaf(xv[c], w.x, acc[0][c]);
      acc[1][c] = fmaf(xv[c], w.y, acc[1][c]);
    }
  }
}

// LayerNorm ("FW-GLM-5-1 l2_p6", self.layer_norm) and the concatenated
// projection [Wq|Wk|Wv|Wg|Wb] ("Kimi-K2.6 l2_p6", op list steps 1-3 and 5-7).
// A block takes 32 cells: one warp per cell normalises it into the
// channel-major operand; then 2-output x 16-cell thread tiles cover the 4D
// main outputs and a last pass the h bias outputs. The bias of cell (b, r, c)
// goes to [b, t, r, c] of the plane, or to [b, t, c, r] for the ending node
// (the plane is indexed [query, key] along the attended line).
__global__ void __launch_bounds__(kProjThreads)
ln_proj_f32(const float* __restrict__ x, long long cells, int N, int D, int h, int ending,
            const float* __restrict__ gamma, const float* __restrict__ beta,
            const float* __restrict__ Wt, int ldw,   // [D][ldw], 4D + h columns used
            const float* __restrict__ bg,
            float* __restrict__ q, float* __restrict__ k, float* __restrict__ v,
            float* __restrict__ g, float* __restrict__ bias) {
  extern __shared__ float xt[];            // [D][kXtLd]
  const long long cell0 = (long long)blockIdx.x * kCellsPerBlock;
  const int ncell = (int)min((long long)kCellsPerBlock, cells - cell0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Mean and biased variance over D, eps 1e-5 inside the square root.
  for (int c = warp; c < kCellsPerBlock; c += kProjThreads / 32) {
    const float* row = x + (cell0 + c) * D;
    const bool real = c < ncell;
    float s = 0.f;
    for (int e = lane; e < D; e += 32) s += real ? row[e] : 0.f;
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float mean = s / D;
    float ss = 0.f;
    for (int e = lane; e < D; e += 32) { const float t = real ? row[e] - mean : 0.f; ss += t * t; }
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rstd = 1.0f / sqrtf(ss / D + 1e-5f);
    for (int e = lane; e < D; e += 32)
      xt[e * kXtLd + c] = real ? (row[e] - mean) * rstd * gamma[e] + beta[e] : 0.f;
  }
  __syncthreads();

  const long long NN = (long long)N * N;
  constexpr int CT = 16;
  const int tiles = (4 * D / 2) * (kCellsPerBlock / CT);
  for (int t = tid; t < tiles; t += kProjThreads) {
    const int o0 = (t / (kCellsPerBlock / CT)) * 2, c0 = (t % (kCellsPerBlock / CT)) * CT;
    float acc[2][CT];
    tile_gemm<CT>(xt, c0, D, Wt, ldw, o0, acc);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int o = o0 + i, sect = o / D, col = o % D;
      float* dst = sect == 0 ? q : sect == 1 ? k : sect == 2 ? v : g;
#pragma unroll
      for (int c = 0; c < CT; ++c) {
        float val = acc[i][c];
        if (sect == 3) val = 1.0f / (1.0f + expf(-(val + bg[col])));
        if (c0 + c < ncell) dst[(cell0 + c0 + c) * D + col] = val;
      }
    }
  }
  // The h bias outputs, bias[b, t, r, c] of each cell.
  for (int i = tid; i < h * kCellsPerBlock; i += kProjThreads) {
    const int t = i / kCellsPerBlock, c = i % kCellsPerBlock;
    float acc = 0.f;
    for (int e = 0; e < D; ++e) acc = fmaf(xt[e * kXtLd + c], Wt[(size_t)e * ldw + 4 * D + t], acc);
    if (c < ncell) {
      const long long cell = cell0 + c, b = cell / NN, rc = cell - b * NN;
      const long long pos = ending ? (rc % N) * N + rc / N : rc;
      bias[(b * h + t) * NN + pos] = acc;
    }
  }
}

// Row attention ("Kimi-K2.6 l2_p6", op list steps 8-16): block = (128 queries
// j, head t, line (b, a)); one thread per query, keys in chunks of KC. Cell x
// of the line is b N^2 + a sa + x sx, (sa, sx) = (N, 1) for the starting node
// and (1, N) for the ending node (END); the pair bias is read at [b, t, query,
// key], and the query-key mask at b N^2 + query sa + key sx.
// Heads wider than 64 take two threads per query (adjacent lanes), each holding
// half of the head's query and accumulator; the two halves of a dot product
// meet through one shuffle. A thread then needs 2 x 64 registers for them
// instead of 2 x 128, which no register file of 255 per thread holds.
template <int MAXD>
constexpr int f32_split() { return MAXD >= 128 ? 2 : 1; }

template <int MAXD, int KC, bool END>
__global__ void __launch_bounds__(kQueriesPerBlock * f32_split<MAXD>())
row_attn_f32(const float* __restrict__ q, const float* __restrict__ k,
             const float* __restrict__ v, const float* __restrict__ bias,
             const int32_t* __restrict__ mask, int mask_mode,
             int N, int D, int h, int d, float* __restrict__ o) {
  const int sa = END ? 1 : N, sx = END ? N : 1;
  __shared__ float Ks[KC][MAXD];
  __shared__ float Vs[KC][MAXD];
  __shared__ float Bs[kQueriesPerBlock][KC + 1];
  __shared__ unsigned char Ms[kQueriesPerBlock][KC + 1];
  __shared__ int Mrow[KC];

  constexpr int SPLIT = f32_split<MAXD>();       // threads per query
  constexpr int HD = MAXD / SPLIT;               // head channels per thread
  constexpr int NT = kQueriesPerBlock * SPLIT;   // threads per block
  const int tid = threadIdx.x / SPLIT;           // the query of the block
  const int part = threadIdx.x % SPLIT;          // channels part * HD .. + HD - 1
  const long long row = blockIdx.x;              // b * N + a
  const int t = blockIdx.y;
  const long long b = row / N;
  const long long line0 = b * (long long)N * N + (row - b * N) * sa;   // cell 0 of the line
  const int j0 = blockIdx.z * kQueriesPerBlock;
  const int j = j0 + tid;
  const bool active = j < N;
  const long long NN = (long long)N * N;
  const float scale = 1.0f / sqrtf((float)d);

  float qv[HD], acc[HD];
#pragma unroll
  for (int e = 0; e < HD; ++e) {
    const int ee = part * HD + e;
    qv[e] = (active && ee < d) ? q[(line0 + (long long)j * sx) * D + t * d + ee] : 0.f;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;

  for (int k0 = 0; k0 < N; k0 += KC) {
    const int nk = min(KC, N - k0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < KC * MAXD; idx += NT) {
      const int kk = idx / MAXD, e = idx % MAXD;
      const bool in = kk < nk && e < d;
      const long long src = (line0 + (long long)(k0 + kk) * sx) * D + t * d + e;
      Ks[kk][e] = in ? k[src] : 0.f;
      Vs[kk][e] = in ? v[src] : 0.f;
    }
    for (int idx = threadIdx.x; idx < kQueriesPerBlock * KC; idx += NT) {
      const int jj = idx / KC, kk = idx % KC;
      const bool in = (j0 + jj) < N && kk < nk;
      Bs[jj][kk] = in ? bias[(b * h + t) * NN + (long long)(j0 + jj) * N + k0 + kk] : 0.f;
      if (mask_mode == TRI_ATTN_MASK_QUERY_KEY)
        Ms[jj][kk] =
            (in && mask[b * NN + (long long)(j0 + jj) * sa + (long long)(k0 + kk) * sx] != 0) ? 1 : 0;
    }
    if (mask_mode == TRI_ATTN_MASK_ROW_KEY && threadIdx.x < KC)
      Mrow[threadIdx.x] = (int)threadIdx.x < nk ? mask[line0 + (long long)(k0 + threadIdx.x) * sx] : 0;
    __syncthreads();

    // Keys four at a time: four independent dot-product chains, one rescale.
#pragma unroll 1
    for (int kk = 0; kk < nk; kk += 4) {
      float lg[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < HD; ++e) dot = fmaf(qv[e], Ks[kk + u][part * HD + e], dot);   // KC % 4 == 0
        if constexpr (SPLIT == 2) dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        float v = dot * scale + Bs[tid][kk + u];
        const int keep = mask_mode == TRI_ATTN_MASK_ROW_KEY ? Mrow[kk + u] : Ms[tid][kk + u];
        if (!keep) v = -1e9f;                     // replacement by -1e9
        lg[u] = kk + u < nk ? v : -INFINITY;      // past N: weight 0
      }
      const float mn = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
      if (mn > m) {                               // running maximum moved: rescale
        const float alpha = expf(m - mn);         // exp(-inf) = 0 before the first key
        l *= alpha;
#pragma unroll
        for (int e = 0; e < HD; ++e) acc[e] *= alpha;
        m = mn;
      }
      float pk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        pk[u] = expf(lg[u] - m);
        l += pk[u];
      }
#pragma unroll
      for (int e = 0; e < HD; ++e) {
        const int ee = part * HD + e;
        acc[e] = fmaf(pk[3], Vs[kk + 3][ee], fmaf(pk[2], Vs[kk + 2][ee],
                 fmaf(pk[1], Vs[kk + 1][ee], fmaf(pk[0], Vs[kk][ee], acc[e]))));
      }
    }
  }
  if (active) {
    const float inv = 1.0f / l;
#pragma unroll
    for (int e = 0; e < HD; ++e)
      if (part * HD + e < d) o[(line0 + (long long)j * sx) * D + t * d + part * HD + e] = acc[e] * inv;
  }
}

// Gate and output projection ("Kimi-K2.6 l2_p6", op list steps 17-18): the
// block's 32 cells of g * o go channel-major into shared memory, then
// 2-output x 8-cell thread tiles of the output projection.
__global__ void __launch_bounds__(kProjThreads)
gate_out_f32(const float* __restrict__ g, const float* __restrict__ o, long long cells, int D,
             const float* __restrict__ Wot,     // [D][D] (in, out)
             const float* __restrict__ bo, float* __restrict__ out) {
  extern __shared__ float xt[];               // [D][kXtLd]
  const long long cell0 = (long long)blockIdx.x * kCellsPerBlock;
  const int ncell = (int)min((long long)kCellsPerBlock, cells - cell0);
  for (int idx = threadIdx.x; idx < kCellsPerBlock * D; idx += kProjThreads) {
    const int c = idx / D, e = idx % D;
    const long long src = (cell0 + c) * D + e;
    xt[e * kXtLd + c] = (c < ncell) ? g[src] * o[src] : 0.f;
  }
  __syncthreads();
  constexpr int CT = 8;
  const int tiles = (D / 2) * (kCellsPerBlock / CT);
  for (int t = threadIdx.x; t < tiles; t += kProjThreads) {
    const int o0 = (t / (kCellsPerBlock / CT)) * 2, c0 = (t % (kCellsPerBlock / CT)) * CT;
    float acc[2][CT];
    tile_gemm<CT>(xt, c0, D, Wot, D, o0, acc);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int c = 0; c < CT; ++c)
        if (c0 + c < ncell) out[(cell0 + c0 + c) * D + o0 + i] = acc[i][c] + bo[o0 + i];
  }
}

// The three kernels of one forward on packed weights and the given buffers.
struct F32Launch {
  long long cells;
  int B, N, D, h, mask_mode;
  bool ending;
  const float *x, *gamma, *beta, *w_proj, *bg, *w_out, *bo;
  const int32_t* mask;
  float *q, *k, *v, *g, *o, *bias, *out;
};

cudaError_t launch_f32(const F32Launch& a, cudaStream_t s, tri_attn_s* timing) {
  const int D = a.D, h = a.h, d = a.D / a.h, N = a.N;
  const unsigned nblk = (unsigned)((a.cells + kCellsPerBlock - 1) / kCellsPerBlock);
  const size_t smem = (size_t)kXtLd * D * sizeof(float);
  if (timing) tri_mark(timing, s, 0, nullptr);
  ln_proj_f32<<<nblk, kProjThreads, smem, s>>>(a.x, a.cells, N, D, h, a.ending ? 1 : 0, a.gamma,
                                               a.beta, a.w_proj, proj_ld(D, h), a.bg, a.q, a.k,
                                               a.v, a.g, a.bias);
  if (timing) tri_mark(timing, s, 1, "ln_proj_f32");
  dim3 grid((unsigned)(a.B * (long long)N), h, (N + kQueriesPerBlock - 1) / kQueriesPerBlock);
#define TRI_ATTN_F32_CASE(MD)                                                              \
  case MD:                                                                                 \
    if (a.ending)                                                                          \
      row_attn_f32<MD, (MD >= 128 ? 16 : kKeyChunk), true>                                \
          <<<grid, kQueriesPerBlock * f32_split<MD>(), 0, s>>>(                            \
          a.q, a.k, a.v, a.bias, a.mask, a.mask_mode, N, D, h, d, a.o);                    \
    else                                                                                   \
      row_attn_f32<MD, (MD >= 128 ? 16 : kKeyChunk), false>                               \
          <<<grid, kQueriesPerBlock * f32_split<MD>(), 0, s>>>(                            \
          a.q, a.k, a.v, a.bias, a.mask, a.mask_mode, N, D, h, d, a.o);                    \
    break;
  const int md = d <= 8 ? 8 : d <= 16 ? 16 : d <= 32 ? 32 : d <= 64 ? 64 : 128;
  switch (md) {
    TRI_ATTN_F32_CASE(8)
    TRI_ATTN_F32_CASE(16)
    TRI_ATTN_F32_CASE(32)
    TRI_ATTN_F32_CASE(64)
    TRI_ATTN_F32_CASE(128)
  }
#undef TRI_ATTN_F32_CASE
  if (timing) tri_mark(timing, s, 2, "row_attn_f32");
  gate_out_f32<<<nblk, kProjThreads, smem, s>>>(a.g, a.o, a.cells, D, a.w_out, a.bo, a.out);
  if (timing) tri_mark(timing, s, 3, "gate_out_f32");
  return cudaGetLastError();
}

}  // namespace

cudaError_t tri_f32_pack_weights(tri_attn_s* t, const void* Wq, const void* Wk, const void* Wv,
                                 const void* Wg, const void* Wb, const void* Wo,
                                 cudaStream_t s) {
  const int D = t->D, h = t->h, nout = proj_ld(D, h);
  float* wp = (float*)t->w_proj;
  const void* mats[5] = {Wq, Wk, Wv, Wg, Wb};
  for (int m = 0; m < 5; ++m) {
    const int rows = m < 4 ? D : h;
    const int n = rows * D;
    pack_transpose_f32<<<(n + 255) / 256, 256, 0, s>>>((const float*)mats[m], rows, D, wp, nout,
                                                       m * D);
  }
  pack_transpose_f32<<<(D * D + 255) / 256, 256, 0, s>>>((const float*)Wo, D, D,
                                                         (float*)t->w_out, D, 0);
  return cudaGetLastError();
}

cudaError_t tri_f32_forward(tri_attn_s* t, cudaStream_t s, const float* x,
                            const int32_t* mask, float* out) {
  F32Launch a;
  a.cells = t->cells; a.B = t->B; a.N = t->N; a.D = t->D; a.h = t->h;
  a.mask_mode = t->mask_mode; a.ending = t->ending;
  a.x = x; a.gamma = t->gamma; a.beta = t->beta; a.w_proj = (const float*)t->w_proj;
  a.bg = t->bg; a.w_out = (const float*)t->w_out; a.bo = t->bo; a.mask = mask;
  a.q = (float*)t->q; a.k = (float*)t->k; a.v = (float*)t->v; a.g = (float*)t->g;
  a.o = (float*)t->o; a.bias = t->bias; a.out = out;
  return launch_f32(a, s, t);
}

cudaError_t tri_f32_forward_raw(const TriF32Raw& r, cudaStream_t s) {
  const int D = r.D, h = r.h, nout = proj_ld(D, h);
  const void* mats[5] = {r.Wq, r.Wk, r.Wv, r.Wg, r.Wb};
  for (int m = 0; m < 5; ++m) {
    const int rows = m < 4 ? D : h;
    const int n = rows * D;
    pack_transpose_f32<<<(n + 255) / 256, 256, 0, s>>>((const float*)mats[m], rows, D, r.w_proj,
                                                       nout, m * D);
  }
  pack_transpose_f32<<<(D * D + 255) / 256, 256, 0, s>>>(r.Wo, D, D, r.w_out, D, 0);
  F32Launch a;
  a.cells = (long long)r.B * r.N * r.N; a.B = r.B; a.N = r.N; a.D = D; a.h = h;
  a.mask_mode = r.mask_mode; a.ending = r.ending;
  a.x = r.x; a.gamma = r.gamma; a.beta = r.beta; a.w_proj = r.w_proj; a.bg = r.bg;
  a.w_out = r.w_out; a.bo = r.bo; a.mask = r.mask;
  a.q = r.q; a.k = r.k; a.v = r.v; a.g = r.g; a.o = r.o; a.bias = r.bias; a.out = r.out;
  return launch_f32(a, s, nullptr);
}
