// bf16 tensor-core path of triangular self-attention, starting and ending node
// (sm_103a).
//
// Four kernels; the three GEMM-shaped ones are built on tcgen05 MMAs with
// operands staged by TMA in swizzled shared memory and accumulators in tensor
// memory (TMEM):
//
//   ln_proj_tc   LayerNorm as the prologue of one concatenated projection GEMM
//                x_hat [128 cells x 128] . [Wq|Wk|Wv|Wg]^T -> 512 TMEM columns;
//                the epilogue writes q, k, v and sigmoid(g + bg) in bf16. The
//                h pair-bias outputs (Wb x_hat, with gamma and beta folded into
//                Wb) come out of the LayerNorm's statistics pass on the CUDA
//                cores and go, scaled by log2(e), to an fp32 plane in cell
//                order.
//   bias_rows    the attention's fp16 bias plane (B, h, N, Nb), indexed
//                [query, key] along the attended line: each (head, query) row
//                minus its largest entry (the softmax is unchanged, and fp16
//                is then precise where the weights are large).
//   mask_summary / mask_summary_cols
//                keep bits and a "keeps some key" flag of every line.
//   row_attn_tc  flash-style line attention, persistent: a work unit is
//                (b, head t, R = 3 lines, 128 queries) streaming 64-key tiles.
//                Lines are grid rows (starting node) or columns (ending node);
//                only the tensor maps tell them apart. S = Q K^T goes to TMEM;
//                one softmax warpgroup per line adds the shared fp16 bias
//                tile, drops masked keys and writes P = 2^(x - mu) in bf16
//                over S (mu: a lazily moved reference max); O += P V
//                accumulates in TMEM. The (B, N, h, N, N) logits never exist.
//   gate_out_tc  g * o formed in shared memory as the A operand of the output
//                projection GEMM; the epilogue adds bo and stores bf16. Tiles
//                are 128 cells in memory order, or 128 rows of one grid
//                column (the host-buffer forward of the ending node).
//
// The file ends with the host side: tensor maps, launchers, the device-buffer
// forward and the host-buffer pipeline that overlaps the host copies with
// chunks of the same kernels.
//
// Passages followed: POPCORNBENCH "Kimi-K2.6 l2_p6", forward op list steps
// 1-18 and layer definitions; "FW-GLM-5-1 l2_p6", quoted Model.forward.
#include <math.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Shared helpers
// ---------------------------------------------------------------------------

struct Abort {
  int* flag;              // shared-memory flag: nonzero once any role gave up
  unsigned int* dev_err;  // handle's device error word
  long long polls;        // poll cap of ordinary waits
};

// Bounded wait; on time-out or when another role has already aborted, raises
// the abort flag (and records a time-out) and returns false.
__device__ __forceinline__ bool wait_or_abort_slow(uint64_t* bar, uint32_t parity, const Abort a);
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const Abort& a) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  return wait_or_abort_slow(bar, parity, a);
}
__device__ __forceinline__ bool wait_or_abort_slow(uint64_t* bar, uint32_t parity, const Abort a) {
  const uint64_t t0 = tc::global_timer_ns();
  for (long long n = 1; n < a.polls; ++n) {
    // Sleeps up to 20 us per poll instead of spinning; the phase wakes it.
    if (tc::mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if (tc::lds_volatile(a.flag)) return false;
    if ((n & 15) == 0 && tc::global_timer_ns() - t0 > 2000000000ull) break;
  }
  *(volatile int*)a.flag = 1;
  atomicOr(a.dev_err, TRI_DEV_ERR_TIMEOUT);
  return false;
}

// Warp-uniform form for warps that go on to issue warp-collective tcgen05
// loads: every lane waits, and the warp proceeds only if all lanes succeeded.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, const Abort& a) {
  const bool ok = wait_or_abort(bar, parity, a);
  return __all_sync(0xffffffffu, ok);
}

// Drain wait used at teardown: ignores the abort flag and the poll cap so that
// copies and MMAs still in flight land before the CTA releases its memory.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  tc::mbar_wait(bar, parity, 1ll << 40);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Logistic function for the gate, 1/(1 + e^-z) = (1 + tanh(z/2)) / 2, with the
// hardware tanh approximation (one special-function operation; its error is
// well below the bf16 rounding the gate gets).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_approx(float z) {
  return fmaf(0.5f, tanh_approx(0.5f * z), 0.5f);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// fp16 half of a packed pair plus an fp32 value, rounded once in fp32.
__device__ __forceinline__ float add_f16lo_f32(uint32_t h2, float c) {
  float d;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, lo, %2;\n\t}"
      : "=f"(d) : "r"(h2), "f"(c));
  return d;
}
__device__ __forceinline__ float add_f16hi_f32(uint32_t h2, float c) {
  float d;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.f16 %0, hi, %2;\n\t}"
      : "=f"(d) : "r"(h2), "f"(c));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// ---------------------------------------------------------------------------
// K1: LayerNorm + concatenated projection
// ---------------------------------------------------------------------------
namespace k1 {
constexpr int BM = 128;                 // cells per tile
constexpr int KD = 128;                 // channels (GEMM K)
constexpr int NQ = 512;                 // q|k|v|g columns
// Warps 0-7 LayerNorm (two per row: warp q handles channel half 0 of rows
// 32q..32q+31, warp q + 4 half 1), warps 8-15 epilogue (two per TMEM lane
// quarter, one per column half), warp 16 TMA, warp 17 MMA. The LayerNorm of
// the next tile runs while the epilogue drains the current one.
constexpr int kWorkers = 256;           // LayerNorm threads (and epilogue threads)
constexpr int kThreads = 2 * kWorkers + 64;
constexpr int kTmaWarp = 16, kMmaWarp = 17;
constexpr uint32_t W_BYTES = NQ * KD * 2;           // 128 KB, two K-halves of 64 KB
constexpr uint32_t X_BYTES = BM * KD * 2;           // 32 KB, two K-halves of 16 KB
constexpr uint32_t OFF_W = 0;
constexpr uint32_t OFF_X = OFF_W + W_BYTES;
constexpr uint32_t OFF_STG = OFF_X + 2 * X_BYTES;   // per worker warp: 2 x (32 rows x 64 B)
constexpr uint32_t STG_BYTES = 32 * 64;
constexpr uint32_t OFF_BAR = OFF_STG + 8 * 2 * STG_BYTES;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;     // + alignment slack

// The two worker warps of lane quarter q (q and q + 4), which share the tile's
// rows, meet at named barrier 1 + q.
__device__ __forceinline__ void pair_sync(int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
}

struct Bars {
  uint64_t w_full, x_full[2], x_empty[2], a_ready[2], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort;
};

// LayerNorm and bias parameters travel by value in the kernel parameter block
// (constant bank): every read index is known at compile time.
// gw[t][c] = gamma[c] Wb[t][c], gws[t] = sum_c gw[t][c], bw[t] = sum_c beta[c] Wb[t][c]:
// with t_c = (x_c - mean) rstd, bias[t] = sum_c x_hat_c Wb[t][c]
// = rstd (sum_c (x_c - K) gw[t][c] - (mean - K) gws[t]) + bw[t] for any shift K.
struct alignas(16) Consts {     // 16-byte aligned: rows are read as float2 pairs
  float gamma[KD], beta[KD], bg[KD], gw[4][KD], gws[4], bw[4];
};
static_assert(offsetof(Consts, gw) % 16 == 0 && offsetof(Consts, beta) % 16 == 0,
              "parameter rows must stay 8-byte aligned");

struct Params {
  long long cells;
  int N, h, mask_mode, ntiles;       // this launch: tiles tile0 .. tile0 + ntiles - 1
  int tile0;
  const int32_t* mask;
  __nv_bfloat16 *q, *k, *v, *g;
  float* bias32;               // (B, h, N, N) fp32 in cell order, scaled by log2(e)
  unsigned int* dev_err;
  long long polls;
  float q_scale;               // q is stored times log2(e) / sqrt(d)
};

// Persistent: CTA c serves 128-cell tiles c, c + G, ... [Wq;Wk;Wv;Wg] (bf16,
// K-major, 128 KB) stays in shared memory. Per tile the x tile arrives by TMA;
// the 256 workers normalise it in place (the two threads of a cell each own
// one 64-channel half; each takes the row statistics and two of the h = 4
// bias outputs from the whole row in one shifted pass, the bias through gamma
// and beta folded into Wb); the MMA warp
// issues the two N = 256 halves (q|k, v|g) into TMEM columns 0-255 / 256-511,
// each with its own full/empty barriers, so the next tile's first half can
// start while the epilogue still reads the second.
__global__ void __launch_bounds__(kThreads, 1)
ln_proj_tc(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
           const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
           const Params p, const __grid_constant__ Consts cst) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = (Bars*)(smem + OFF_BAR);
  const float* s_bg = cst.bg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Abort ab{&bars->abort, p.dev_err, p.polls};

  if (tid == 0) {
    tc::mbar_init(&bars->w_full, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars->x_full[b], 1);
      tc::mbar_init(&bars->x_empty[b], 1);
      tc::mbar_init(&bars->a_ready[b], kWorkers);
      tc::mbar_init(&bars->acc_full[b], 1);
      tc::mbar_init(&bars->acc_empty[b], kWorkers);
    }
    tc::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int my_tiles = 0;
  for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) ++my_tiles;
  int issued = 0;                          // tile loads issued (producer thread)

  if (warp == kTmaWarp) {
    // ---------------- TMA producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&map_x);
      tc::tma_prefetch_desc(&map_w);
      tc::mbar_arrive_expect_tx(&bars->w_full, W_BYTES);
      for (int kh = 0; kh < 2; ++kh)
        for (int nh = 0; nh < 2; ++nh)
          tc::tma_load_2d(smem + OFF_W + kh * 65536 + nh * 32768, &map_w, &bars->w_full,
                          kh * 64, nh * 256);
      for (int it = 0; it < my_tiles; ++it) {
        const int b = it & 1;
        if (it >= 2 && !wait_or_abort(&bars->x_empty[b], ((it >> 1) - 1) & 1, ab)) break;
        const int tile = p.tile0 + blockIdx.x + it * gridDim.x;
        uint8_t* xs = smem + OFF_X + b * X_BYTES;
        tc::mbar_arrive_expect_tx(&bars->x_full[b], X_BYTES);
        tc::tma_load_2d(xs, &map_x, &bars->x_full[b], 0, tile * BM);
        tc::tma_load_2d(xs + 16384, &map_x, &bars->x_full[b], 64, tile * BM);
        issued = it + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 256, 0, 0);
      const uint32_t w0 = tc::smem_addr(smem + OFF_W);
      bool ok = wait_or_abort(&bars->w_full, 0, ab);
      for (int it = 0; ok && it < my_tiles; ++it) {
        const int b = it & 1;
        if (!wait_or_abort(&bars->a_ready[b], (it >> 1) & 1, ab)) break;
        const uint32_t a0 = tc::smem_addr(smem + OFF_X + b * X_BYTES);
        for (int nh = 0; nh < 2 && ok; ++nh) {
          if (it >= 1 && !wait_or_abort(&bars->acc_empty[nh], (it - 1) & 1, ab)) { ok = false; break; }
          tc::tc_fence_after();
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ko = (ks >> 2) * 16384 + (ks & 3) * 32;
            const uint64_t ad = tc::smem_desc(a0 + ko, 16, 1024, tc::SWZ_128B);
            const uint64_t bd = tc::smem_desc(w0 + (ks >> 2) * 65536 + nh * 32768 + (ks & 3) * 32,
                                              16, 1024, tc::SWZ_128B);
            tc::mma_bf16_ss(tmem + nh * 256, ad, bd, idesc, ks > 0);
          }
          tc::mma_commit(&bars->acc_full[nh]);
        }
        if (!ok) break;
        tc::mma_commit(&bars->x_empty[b]);
      }
      tc::mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0);
    }
  } else if (warp < kWorkers / 32) {
    // ---------------- LayerNorm: cell row r, channel half hh
    const int q4 = warp & 3, hh = warp >> 2;
    const int r = q4 * 32 + lane;
    // Parameter pairs (one 8-byte constant load each): this thread's two bias
    // heads and the LayerNorm affine.
    const float2* gw2[2] = {(const float2*)cst.gw[2 * hh], (const float2*)cst.gw[2 * hh + 1]};
    const float2* gamma2 = (const float2*)cst.gamma;
    const float2* beta2 = (const float2*)cst.beta;
    const long long NN = (long long)p.N * p.N;
    bool ok = true;
    for (int it = 0; ok && it < my_tiles; ++it) {
      const int b = it & 1;
      if (!warp_wait_or_abort(&bars->x_full[b], (it >> 1) & 1, ab)) { ok = false; break; }
      const int tile = p.tile0 + blockIdx.x + it * gridDim.x;
      const long long cell = (long long)tile * BM + r;
      uint8_t* xs = smem + OFF_X + b * X_BYTES;
      auto chunk = [&](int c) -> uint4 {
        return *(const uint4*)(xs + (c >> 3) * 16384 + tc::swz_offset(r, c & 7, 128));
      };
      // One pass over the whole row, shifted by its first channel K so that the
      // sums do not cancel: the row statistics and this thread's two bias heads
      // (2 hh, 2 hh + 1) through the folded constants of k1::Consts.
      const float K0 = bf16_lo(chunk(0).x);
      const float2 nk2 = make_float2(-K0, -K0);
      float2 s2 = make_float2(0.f, 0.f), q2 = make_float2(0.f, 0.f);
      float2 bp[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 u = chunk(c);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i0 = c * 8 + 2 * e;
          const float2 d = __fadd2_rn(make_float2(bf16_lo(w4[e]), bf16_hi(w4[e])), nk2);
          s2 = __fadd2_rn(s2, d);
          q2 = __ffma2_rn(d, d, q2);
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2)
            bp[t2] = __ffma2_rn(d, gw2[t2][i0 / 2], bp[t2]);
        }
      }
      const float S1 = (s2.x + s2.y) * (1.0f / KD);             // mean of x - K
      const float var = fmaxf((q2.x + q2.y) * (1.0f / KD) - S1 * S1, 0.f);
      const float mean = K0 + S1;
      const float rstd = rsqrtf(var + 1e-5f);
      float bsum[2];
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2)
        bsum[t2] = rstd * ((bp[t2].x + bp[t2].y) - S1 * cst.gws[2 * hh + t2]) + cst.bw[2 * hh + t2];
      // Normalise this thread's half, rounded to bf16 as the MMA sees it.
      const float2 rs2 = make_float2(rstd, rstd), nm2 = make_float2(-mean * rstd, -mean * rstd);
      uint32_t mine[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 u = chunk(hh * 8 + c);
        const uint32_t in4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i0 = hh * 64 + c * 8 + 2 * e;
          const float2 t = __ffma2_rn(make_float2(bf16_lo(in4[e]), bf16_hi(in4[e])), rs2, nm2);
          const float2 y = __ffma2_rn(t, gamma2[i0 / 2], beta2[i0 / 2]);
          mine[c * 4 + e] = tc::pack_bf16x2(y.x, y.y);
        }
      }
      // The other thread of this row has read both halves once it reaches the
      // pair barrier; then each thread writes its own half back.
      pair_sync(q4);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *(uint4*)(xs + hh * 16384 + tc::swz_offset(r, c, 128)) =
            make_uint4(mine[4 * c], mine[4 * c + 1], mine[4 * c + 2], mine[4 * c + 3]);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars->a_ready[b]);
      if (cell < p.cells) {
        // The pair bias of the cell, in cell order (consecutive threads,
        // consecutive cells): bias_rows turns the plane into the attention's
        // [query, key] layout.
        const long long bb = cell / NN;
        const long long rc = cell - bb * NN;
        bool keep = true;
        if (p.mask_mode == TRI_ATTN_MASK_QUERY_KEY) keep = p.mask[cell] != 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int head = 2 * hh + t;
          if (head < p.h)
            p.bias32[(bb * p.h + head) * NN + rc] = keep ? bsum[t] * kLog2e : -INFINITY;
        }
      }
    }
  } else if (warp < 2 * kWorkers / 32) {
    // ---------------- epilogue: cell row r = TMEM lane, column half hh
    const int ew = warp - kWorkers / 32;
    const int q4 = ew & 3, hh = ew >> 2;
    // Epilogue: each 32-row x 32-column chunk goes TMEM -> registers -> bf16 in a
    // swizzled smem staging tile -> one TMA store (full 64-byte row segments;
    // rows past the last cell are clipped by the tensor bounds).
    // The two warps of a lane quarter split every 128-column section (q, k, v,
    // g) in halves, so both carry the same sigmoid load; accumulator half nh
    // (q|k or v|g) is released as soon as both warps have read it.
    uint8_t* stg0 = smem + OFF_STG + ew * 2 * STG_BYTES;
    int nst = 0;                                  // TMA stores issued by this warp
    auto epilogue = [&](int it) -> bool {
      const int tile = p.tile0 + blockIdx.x + it * gridDim.x;
      const int row0 = tile * BM + q4 * 32;
#pragma unroll 1
      for (int nh = 0; nh < 2; ++nh) {
        if (!warp_wait_or_abort(&bars->acc_full[nh], it & 1, ab)) return false;
        tc::tc_fence_after();
        // Half-chunk k (16 columns) of the 8 this warp drains from accumulator
        // half nh: chunk k / 2 = 32 columns of section nh * 2 + k / 4. The load
        // of half-chunk k + 1 is in flight while half-chunk k is converted.
        auto hc_addr = [&](int k) {
          const int cc = k >> 1, sect = nh * 2 + (cc >> 1);
          return tc::tmem_addr(tmem, q4 * 32, sect * 128 + hh * 64 + (cc & 1) * 32 + (k & 1) * 16);
        };
        uint32_t accb[2][16];
        tc::tmem_ld16(hc_addr(0), accb[0]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int cc = k >> 1;
          const int sect = nh * 2 + (cc >> 1);
          const int col0 = hh * 64 + (cc & 1) * 32;          // within the section
          tc::tmem_ld_wait();
          if (k + 1 < 8) tc::tmem_ld16(hc_addr(k + 1), accb[(k + 1) & 1]);
          const uint32_t (&acc)[16] = accb[k & 1];
          uint32_t packed[8];
          if (sect == 3) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int cg = col0 + (k & 1) * 16 + 2 * e;
              const float z0 = __uint_as_float(acc[2 * e]) + s_bg[cg];
              const float z1 = __uint_as_float(acc[2 * e + 1]) + s_bg[cg + 1];
              packed[e] = tc::pack_bf16x2(sigmoid_approx(z0), sigmoid_approx(z1));
            }
          } else if (sect == 0) {
            // q leaves in the log2 domain of the attention's exponentials,
            // scaled by log2(e) / sqrt(d) before its one rounding to bf16.
#pragma unroll
            for (int e = 0; e < 8; ++e)
              packed[e] = tc::pack_bf16x2(__uint_as_float(acc[2 * e]) * p.q_scale,
                                          __uint_as_float(acc[2 * e + 1]) * p.q_scale);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              packed[e] = tc::pack_bf16x2(__uint_as_float(acc[2 * e]), __uint_as_float(acc[2 * e + 1]));
          }
          uint8_t* stg = stg0 + (nst & 1) * STG_BYTES;
          if ((k & 1) == 0 && nst >= 2) {    // the store two back has read this staging tile
            if (lane == 0) tc::tma_store_wait_read<1>();
            __syncwarp();
          }
#pragma unroll
          for (int c = 0; c < 2; ++c)
            *(uint4*)(stg + tc::swz_offset(lane, (k & 1) * 2 + c, 64)) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          if (k & 1) {
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const CUtensorMap* m = sect == 0 ? &map_q : sect == 1 ? &map_k : sect == 2 ? &map_v : &map_g;
              tc::tma_store_2d(m, stg, col0, row0);
              tc::tma_store_commit();
            }
            ++nst;
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&bars->acc_empty[nh]);
      }
      return true;
    };
    for (int it = 0; it < my_tiles; ++it)
      if (!epilogue(it)) break;
  }

  // ---------------- teardown: every issued copy lands, every MMA completes
  if (warp >= kWorkers / 32 && warp < 2 * kWorkers / 32 && lane == 0) tc::tma_store_wait_all<0>();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kTmaWarp && lane == 0) {
    drain_wait(&bars->w_full, 0);
    for (int it = issued - 1; it >= 0 && it >= issued - 2; --it)
      drain_wait(&bars->x_full[it & 1], (it >> 1) & 1);
  }
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 512);
}
}  // namespace k1


// ---------------------------------------------------------------------------
// K2: flash row attention
// ---------------------------------------------------------------------------
namespace k2 {
constexpr int R = 3;                    // lines per work unit = softmax warpgroups
constexpr int BQ = 128;                 // queries j per unit
constexpr int BK = 64;                  // keys per sub-tile (one S buffer)
constexpr int KVK = 128;                // keys per K/V stage (two sub-tiles)
constexpr int DH = 32;                  // head dim
constexpr int KV_STAGES = 2;
constexpr int B_STAGES = 3;
constexpr int kIssuers = R;             // MMA issuer warps, one line each
constexpr int kSoftmaxWarps = 4 * R;
// Warpgroup 0: warp 0 TMA, warp 1 + r issues the MMAs of line r (both roles
// run as whole warps; one elected lane issues); warpgroup w = 1..3 runs the
// softmax of line w - 1. Registers move from the control warpgroup to the
// softmax ones: 512 x 128 >= 128 x 48 + 384 x 152.
constexpr int kThreads = 512;
constexpr int kRegsCtl = 48, kRegsSoftmax = 152;
// TMEM per line: S0 | S1 (64 fp32 columns each) | O (32). Sub-tile c's S lands
// in buffer c & 1 and its P (bf16 pairs, 32 columns) is written over it; the
// MMA warp issues P V(c) and then S(c + 2) into the same buffer, so the tensor
// pipe's issue order keeps them apart.
constexpr int kTmemPerRow = 160;
constexpr int TM_S1 = 64, TM_O = 128;
constexpr uint32_t Q_BYTES = BQ * DH * 2;            // 8 KB per line
constexpr uint32_t KVT_BYTES = KVK * DH * 2;         // 8 KB: K or V of one line, 128 keys
constexpr uint32_t KV_STAGE = R * 2 * KVT_BYTES;     // 48 KB: [R] K then V
constexpr uint32_t HALF_KV = BK * DH * 2;            // 4 KB: one sub-tile inside a K/V tile
constexpr uint32_t BIAS_BYTES = BQ * BK * 2;         // 16 KB fp16 bias sub-tile
constexpr uint32_t OST_BYTES = 32 * DH * 2;          // 2 KB o staging per softmax warp
constexpr uint32_t OFF_Q = 0;                        // [2][R] Q tiles
constexpr uint32_t OFF_KV = OFF_Q + 2 * R * Q_BYTES;
constexpr uint32_t OFF_BIAS = OFF_KV + KV_STAGES * KV_STAGE;
constexpr uint32_t OFF_OST = OFF_BIAS + B_STAGES * BIAS_BYTES;
constexpr uint32_t OFF_BAR = OFF_OST + kSoftmaxWarps * OST_BYTES;
constexpr uint32_t SMEM = OFF_BAR + 512 + 1024;
static_assert(OFF_KV % 1024 == 0 && OFF_BIAS % 1024 == 0 && OFF_OST % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");

struct Bars {
  uint64_t q_full[2], q_empty[2], kv_full[KV_STAGES], kv_empty[KV_STAGES];
  uint64_t b_full[B_STAGES], b_empty[B_STAGES];
  // s_ready and p_full follow the S/P buffer (sub-tile parity): a warp with no
  // live lanes runs ahead, and its arrivals for sub-tile c + 1 must not complete
  // the phase of sub-tile c.
  uint64_t s_ready[R][2], p_full[R][2], p_free[R][2], o_free[R], drain[R];
  uint32_t tmem_base;
  int abort;
};

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
  unsigned int* dev_err;
  long long polls;
  // The same q, k, v and bias plane as raw tensors, for the exact recomputation
  // of a query row whose sums left the fp32 range: element (b, line a, position
  // x, channel e) of q, k or v sits at b * sb + a * sl + x * sx + e.
  const __nv_bfloat16 *q, *k, *v;
  long long sb, sl, sx;
  const float* bias32;            // (B, h, N, N) fp32 cell order, log2(e) * bias, -inf where dropped
  int ending;                     // the key k of query a is cell (k, a) instead of (a, k)
};

struct Unit {
  int b, t, rg, jt, j0;
};

__device__ __forceinline__ Unit decode_unit(int u, const Params& p) {
  Unit un;
  un.jt = u % p.jtiles;
  un.t = (u / p.jtiles) % p.h;
  const int rgb = u / (p.jtiles * p.h);
  un.rg = rgb % p.row_groups;
  un.b = rgb / p.row_groups;
  un.j0 = un.jt * BQ;
  return un;
}

// The unit gridDim.x further on: digit-wise addition with carries (each digit
// of the step is below its radix, so one subtraction per digit suffices).
__device__ __forceinline__ void step_unit(Unit& u, const Params& p) {
  int v = u.jt + p.step.jt;
  int c = v >= p.jtiles;
  u.jt = c ? v - p.jtiles : v;
  v = u.t + p.step.t + c;
  c = v >= p.h;
  u.t = c ? v - p.h : v;
  v = u.rg + p.step.rg + c;
  c = v >= p.row_groups;
  u.rg = c ? v - p.row_groups : v;
  u.b += p.step.b + c;
  u.j0 = u.jt * BQ;
}

// Position in a stream of sub-tiles: global sub-tile c, its unit ui and key
// sub-tile kt, the K/V stage slot and phase, and the bias slot and phase,
// advanced without dividing.
struct SubIt {
  int c, ui, kt, kvs, kvph, bs, bph;
};
__device__ __forceinline__ void advance(SubIt& it, int KT) {
  ++it.c;
  const bool stage_end = (it.kt & 1) || it.kt == KT - 1;
  if (++it.kt == KT) { it.kt = 0; ++it.ui; }
  if (stage_end && ++it.kvs == KV_STAGES) { it.kvs = 0; it.kvph ^= 1; }
  if (++it.bs == B_STAGES) { it.bs = 0; it.bph ^= 1; }
}

// The softmax's position in its sub-tile stream: global sub-tile c, key
// sub-tile kt and the bias slot and phase.
struct SoftIt {
  int c, kt, bs, bph;
};
__device__ __forceinline__ void advance(SoftIt& it, int KT) {
  ++it.c;
  if (++it.kt == KT) it.kt = 0;
  if (++it.bs == B_STAGES) { it.bs = 0; it.bph ^= 1; }
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Real-key bits of word w (keys 32w..32w+31 of a sub-tile with `left` keys left).
__device__ __forceinline__ uint32_t real_bits(int left, int w) {
  const int n = left - 32 * w;
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// The 32 fp16 biases of half hf of a sub-tile row (brow: the row's swizzled
// base, 16-byte chunk q at brow ^ (q << 4)).
__device__ __forceinline__ void load_bias_half(uint32_t brow, int hf, uint4 (&bh)[4]) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) bh[q4] = tc::lds128(brow ^ ((hf * 4 + q4) << 4));
}

// Common path of one 32-key half: P = 2^(S + bias) (S in log2 units, the
// reference mu = 0 and every lane live), packed in bf16 pairs; returns the
// sum of P in two partial sums.
__device__ __forceinline__ float2 p_half_fast(const float2 (&x2)[BK / 2], const uint4 (&bh)[4],
                                              int hf, uint32_t (&pk)[16]) {
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint32_t hw[4] = {bh[q4].x, bh[q4].y, bh[q4].z, bh[q4].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = x2[(hf * 4 + q4) * 4 + e];
      const float2 p2 = make_float2(ex2_approx(add_f16lo_f32(hw[e], x.x)),
                                    ex2_approx(add_f16hi_f32(hw[e], x.y)));
      if (e & 1) sb = __fadd2_rn(sb, p2);
      else sa = __fadd2_rn(sa, p2);
      pk[q4 * 4 + e] = tc::pack_bf16x2(p2.x, p2.y);
    }
  }
  return __fadd2_rn(sa, sb);
}

// P of one 32-key half of a lane that is not live: 1 on every real key of a
// uniform row or query (`w` = that half's real-key bits), else 0.
__device__ __forceinline__ void p_half_const(uint32_t w, uint32_t (&pk)[16]) {
  if (w == 0u || w == 0xffffffffu) {
    const uint32_t v = w ? 0x3F803F80u : 0u;
#pragma unroll
    for (int k = 0; k < 16; ++k) pk[k] = v;
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k)
      pk[k] = (((w >> (2 * k)) & 1u) ? 0x3F80u : 0u) | (((w >> (2 * k + 1)) & 1u) ? 0x3F800000u : 0u);
  }
}

// General path of one 32-key half: P = 2^(S + bias - mu) for a live lane; a
// lane that is not live writes 1 on every real key of a uniform row or query
// (`w` = that half's real-key bits), else 0.
__device__ __forceinline__ float2 p_half(const float2 (&x2)[BK / 2], const uint4 (&bh)[4], int hf,
                                         float mu, bool live, uint32_t w, uint32_t (&pk)[16]) {
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
  if (live) {
    const float2 nmu2 = make_float2(-mu, -mu);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const uint32_t hw[4] = {bh[q4].x, bh[q4].y, bh[q4].z, bh[q4].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 y = __fadd2_rn(x2[(hf * 4 + q4) * 4 + e], nmu2);
        const float2 p2 = make_float2(ex2_approx(add_f16lo_f32(hw[e], y.x)),
                                      ex2_approx(add_f16hi_f32(hw[e], y.y)));
        if (e & 1) sb = __fadd2_rn(sb, p2);
        else sa = __fadd2_rn(sa, p2);
        pk[q4 * 4 + e] = tc::pack_bf16x2(p2.x, p2.y);
      }
    }
  } else {
    p_half_const(w, pk);
  }
  return __fadd2_rn(sa, sb);
}

// A query row whose sum l left [2^-16, 2^100) is recomputed exactly on the
// CUDA cores: its logits reached about +100 in log2 units (P = 2^x with the
// fixed reference 0 loses range), or every key it keeps lies more than 16
// below its (head, query) row's largest bias, which may sit at a key the line
// drops (the row-key reading), where the fp16 plane's rounding is no longer
// small. Two passes over the line's keys, the first for the row max m, the
// second for l = sum 2^(x - m) and o = sum 2^(x - m) v / l, in fp32 with the
// fp32 bias. qrow: the row's q (head t); kl, vl: key 0 of the line's k and v
// (head t), sx: the stride between keys; brow: the bias of the row's key 0 in
// the fp32 cell-order plane and bs the stride between keys; keys come from the
// line's mask bits (row reading; mrow) or from the finite biases (query
// reading, mrow = null: the plane holds -inf for dropped keys). o leaves as 16
// bf16 pairs in the lane's row of the 64-byte-swizzled staging tile at stg.
__device__ __noinline__ void exact_row(const __nv_bfloat16* qrow, const __nv_bfloat16* kl,
                                       const __nv_bfloat16* vl, long long sx,
                                       const float* brow, long long bs, const uint32_t* mrow,
                                       int N, uint8_t* stg, int lane) {
  float q[DH];
#pragma unroll
  for (int e = 0; e < DH; ++e) q[e] = __bfloat162float(qrow[e]);
  float m = -INFINITY;
  for (int kk = 0; kk < N; ++kk) {
    if (mrow && !((__ldg(mrow + (kk >> 5)) >> (kk & 31)) & 1u)) continue;
    const float bb = brow[(long long)kk * bs];
    if (bb == -INFINITY) continue;
    const __nv_bfloat16* kr = kl + (long long)kk * sx;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < DH; ++e) s = fmaf(q[e], __bfloat162float(kr[e]), s);
    m = fmaxf(m, s + bb);
  }
  float l = 0.f, o[DH];
#pragma unroll
  for (int e = 0; e < DH; ++e) o[e] = 0.f;
  for (int kk = 0; kk < N; ++kk) {
    if (mrow && !((__ldg(mrow + (kk >> 5)) >> (kk & 31)) & 1u)) continue;
    const float bb = brow[(long long)kk * bs];
    if (bb == -INFINITY) continue;
    const __nv_bfloat16* kr = kl + (long long)kk * sx;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < DH; ++e) s = fmaf(q[e], __bfloat162float(kr[e]), s);
    const float w = exp2f(s + bb - m);
    l += w;
    const __nv_bfloat16* vr = vl + (long long)kk * sx;
#pragma unroll
    for (int e = 0; e < DH; ++e) o[e] = fmaf(w, __bfloat162float(vr[e]), o[e]);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int qc = 0; qc < 4; ++qc) {
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w4[e] = tc::pack_bf16x2(o[8 * qc + 2 * e] * inv, o[8 * qc + 2 * e + 1] * inv);
    *(uint4*)(stg + tc::swz_offset(lane, qc, 64)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

// Persistent: CTA c serves work units unit0 + c, + G, ... A unit is (b, head
// t, R = 3 lines, 128 queries); it streams 64-key sub-tiles. The K and V tiles
// of the three lines arrive 128 keys at a time (one stage serves two
// sub-tiles); the fp16 bias sub-tile they share has a ring of its own.
// Softmax warpgroup r owns line r; sub-tile c's S = Q K^T lands in the line's
// S buffer c & 1 in log2 units (q carries the factor log2(e)/sqrt(d)), and the
// softmax adds the bias, drops masked keys and writes P = 2^x (bf16) over it
// in one pass; the line's MMA warp then issues O += P V(c) and S(c + 2) into
// the same buffer. The reference of the exponentials is fixed at 0: no max is
// taken, and fp32 and bf16 hold 2^x with full relative precision for
// |x| < ~100, far beyond the logits of layer-normalised activations; a query
// row whose sum l ends outside [2^-16, 2^100) is recomputed exactly in the
// unit epilogue (exact_row). A unit's o = O / l is read and stored after the
// next unit's first sub-tile, which hides the completion of the unit's last
// P V.
__global__ void __launch_bounds__(kThreads, 1)
row_attn_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_b,
            const __grid_constant__ CUtensorMap map_o, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = (Bars*)(smem + OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The abort context is rebuilt from the kernel parameters at each use.
#define ab (Abort{&bars->abort, p.dev_err, p.polls})
  const int N = p.N;
  const int KT = (N + BK - 1) / BK;
  int my_units = 0;
  for (int u = blockIdx.x; u < p.units; u += gridDim.x) ++my_units;

  if (tid == 0) {
    for (int q = 0; q < 2; ++q) {
      tc::mbar_init(&bars->q_full[q], 1);
      tc::mbar_init(&bars->q_empty[q], kIssuers);    // one commit per issuer
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      tc::mbar_init(&bars->kv_full[s], 1);
      tc::mbar_init(&bars->kv_empty[s], kIssuers);
    }
    for (int s = 0; s < B_STAGES; ++s) {
      tc::mbar_init(&bars->b_full[s], 1);
      tc::mbar_init(&bars->b_empty[s], kSoftmaxWarps);   // one arrive per softmax warp
    }
    for (int r = 0; r < R; ++r) {
      for (int b = 0; b < 2; ++b) {
        tc::mbar_init(&bars->s_ready[r][b], 1);
        tc::mbar_init(&bars->p_full[r][b], 128);
        tc::mbar_init(&bars->p_free[r][b], 1);
      }
      tc::mbar_init(&bars->o_free[r], 128);
      tc::mbar_init(&bars->drain[r], 1);
    }
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int q_issued = 0, kv_issued = 0, b_issued = 0;    // producer: loads issued

  if (warp < 4) {
    tc::regs_dec<kRegsCtl>();
    if (warp == 0) {
      // ---------------- TMA producer (whole warp; one elected lane issues)
      if (elect_one()) {
        tc::tma_prefetch_desc(&map_q);
        tc::tma_prefetch_desc(&map_k);
        tc::tma_prefetch_desc(&map_v);
        tc::tma_prefetch_desc(&map_b);
      }
      __syncwarp();
      Unit un = decode_unit(p.unit0 + blockIdx.x, p);
      int kvs = 0, kvph = 0, bs = 0, bph = 0;
      bool ok = true;
      for (int ui = 0; ok && ui < my_units; ++ui, step_unit(un, p)) {
        const int a0 = un.rg * R;
        const int qb = ui & 1;
        if (ui >= 2 && !warp_wait_or_abort(&bars->q_empty[qb], ((ui >> 1) - 1) & 1, ab)) break;
        if (elect_one()) {
          tc::mbar_arrive_expect_tx(&bars->q_full[qb], R * Q_BYTES);
          for (int r = 0; r < R; ++r)
            tc::tma_load_4d(smem + OFF_Q + (qb * R + r) * Q_BYTES, &map_q, &bars->q_full[qb],
                            un.t * DH, un.j0, a0 + r, un.b);
        }
        __syncwarp();
        q_issued = ui + 1;
        for (int kt = 0; kt < KT; ++kt) {
          if ((kt & 1) == 0) {
            if (kv_issued >= KV_STAGES && !warp_wait_or_abort(&bars->kv_empty[kvs], kvph ^ 1, ab)) {
              ok = false;
              break;
            }
            if (elect_one()) {
              uint8_t* st = smem + OFF_KV + kvs * KV_STAGE;
              tc::mbar_arrive_expect_tx(&bars->kv_full[kvs], KV_STAGE);
              for (int r = 0; r < R; ++r) {
                tc::tma_load_4d(st + r * 2 * KVT_BYTES, &map_k, &bars->kv_full[kvs], un.t * DH,
                                kt * BK, a0 + r, un.b);
                tc::tma_load_4d(st + r * 2 * KVT_BYTES + KVT_BYTES, &map_v, &bars->kv_full[kvs],
                                un.t * DH, kt * BK, a0 + r, un.b);
              }
            }
            __syncwarp();
            ++kv_issued;
            if (++kvs == KV_STAGES) { kvs = 0; kvph ^= 1; }
          }
          if (b_issued >= B_STAGES && !warp_wait_or_abort(&bars->b_empty[bs], bph ^ 1, ab)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            tc::mbar_arrive_expect_tx(&bars->b_full[bs], BIAS_BYTES);
            tc::tma_load_3d(smem + OFF_BIAS + bs * BIAS_BYTES, &map_b, &bars->b_full[bs], kt * BK,
                            un.j0, un.b * p.h + un.t);
          }
          __syncwarp();
          ++b_issued;
          if (++bs == B_STAGES) { bs = 0; bph ^= 1; }
        }
      }
    } else {
      // ---------------- MMA issuer of line r = warp - 1 (whole warp; one elected lane issues)
      const int r = warp - 1;
      const uint32_t tr = tmem + r * kTmemPerRow;
      constexpr uint32_t id_qk = tc::idesc_bf16_f32(128, BK, 0, 0);
      constexpr uint32_t id_pv = tc::idesc_bf16_f32(128, DH, 0, 1);
      // Descriptors of this line's first Q tile and first K tile; every other
      // operand sits a multiple of 16 bytes further (the start-address field
      // holds address / 16 and stays below 2^14).
      const uint64_t dq0 = tc::smem_desc(tc::smem_addr(smem + OFF_Q + r * Q_BYTES), 16, 512, tc::SWZ_64B);
      const uint64_t dk0 =
          tc::smem_desc(tc::smem_addr(smem + OFF_KV + r * 2 * KVT_BYTES), 16, 512, tc::SWZ_64B);
      const int total = my_units * KT;     // one item per key sub-tile
      auto qk = [&](const SubIt& it) -> bool {
        const int c = it.c;
        if (it.kt == 0 && !warp_wait_or_abort(&bars->q_full[it.ui & 1], (it.ui >> 1) & 1, ab)) return false;
        if ((it.kt & 1) == 0 && !warp_wait_or_abort(&bars->kv_full[it.kvs], it.kvph, ab)) return false;
        tc::tc_fence_after();
        if (elect_one()) {
          const uint64_t qd = dq0 + (uint64_t)(((it.ui & 1) * R * Q_BYTES) >> 4);
          const uint64_t kd = dk0 + (uint64_t)((it.kvs * KV_STAGE + (it.kt & 1) * HALF_KV) >> 4);
#pragma unroll
          for (int ks = 0; ks < DH / 16; ++ks)
            tc::mma_bf16_ss(tr + (c & 1) * TM_S1, qd + 2 * ks, kd + 2 * ks, id_qk, ks > 0);
          tc::mma_commit(&bars->s_ready[r][c & 1]);
          if (it.kt == KT - 1) tc::mma_commit(&bars->q_empty[it.ui & 1]);
        }
        __syncwarp();
        return true;
      };
      auto pv = [&](const SubIt& it) -> bool {
        const int c = it.c;
        if (!warp_wait_or_abort(&bars->p_full[r][c & 1], (c >> 1) & 1, ab)) return false;
        if (it.kt == 0 && it.ui >= 1 && !warp_wait_or_abort(&bars->o_free[r], (it.ui - 1) & 1, ab))
          return false;
        tc::tc_fence_after();
        if (elect_one()) {
          const uint64_t vd =
              dk0 + (uint64_t)((it.kvs * KV_STAGE + KVT_BYTES + (it.kt & 1) * HALF_KV) >> 4);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            tc::mma_bf16_ts(tr + TM_O, tr + (c & 1) * TM_S1 + ks * 8, vd + 64 * ks, id_pv,
                            (it.kt > 0 || ks > 0) ? 1u : 0u);
          tc::mma_commit(&bars->p_free[r][c & 1]);
          if ((it.kt & 1) || it.kt == KT - 1) tc::mma_commit(&bars->kv_empty[it.kvs]);
        }
        __syncwarp();
        return true;
      };
      bool ok = true;
      SubIt itq{0, 0, 0, 0, 0, 0, 0}, itp{0, 0, 0, 0, 0, 0, 0};
      for (; ok && itq.c < 2 && itq.c < total; advance(itq, KT)) ok = qk(itq);
      for (; ok && itp.c < total; advance(itp, KT)) {
        ok = pv(itp);
        if (ok && itq.c < total) {
          ok = qk(itq);
          advance(itq, KT);
        }
      }
      if (elect_one()) tc::mma_commit(&bars->drain[r]);
      __syncwarp();
      drain_wait(&bars->drain[r], 0);
    }
  } else {
    // ---------------- softmax warpgroups: line r of each unit, thread = query row
    tc::regs_inc<kRegsSoftmax>();
    const int r = (warp >> 2) - 1;
    const int sw = warp - 4;                         // softmax warp index
    const int jr = (warp & 3) * 32 + lane;          // query row of the tile = TMEM lane
    const uint32_t tb = tmem + ((uint32_t)((warp & 3) * 32) << 16) + r * kTmemPerRow;
    // Bias row jr of a stage (128-byte swizzle: 16-byte chunk q of the row sits
    // at chunk q ^ (jr & 7)); the row base is 128-byte aligned.
    const uint32_t brow0 = tc::smem_addr(smem + OFF_BIAS) + jr * 128u + ((jr & 7u) << 4);
    const bool qk_mode = p.mask_mode == TRI_ATTN_MASK_QUERY_KEY;
    // A unit's mask summary: the "keeps some key" flag of this lane's query
    // row (query-key) or of the line (row-key), and the mask row whose bits
    // give the keys this lane keeps. Loaded one unit ahead.
    auto unit_loads = [&](const Unit& nu, unsigned& any, const uint32_t*& mrow) {
      const int nj = nu.j0 + jr, ni = nu.rg * R + r;
      const int mr = qk_mode ? nj : ni;
      // Queries past N produce nothing (their stores are clipped): they count
      // as keeping keys so that they never force the general path.
      any = mr < N ? __ldg(p.row_any + (long long)nu.b * N + mr) : (qk_mode ? 1u : 0u);
      mrow = p.mbits + ((long long)nu.b * N + (mr < N ? mr : 0)) * p.words;
    };
    unsigned nx_any = 0u;
    const uint32_t* nx_mrow = p.mbits;
    if (my_units > 0) unit_loads(decode_unit(p.unit0 + blockIdx.x, p), nx_any, nx_mrow);
    // Unit epilogue: o = O / l once the unit's last P V has landed, staged in
    // shared memory and written by one TMA store per warp (queries past N are
    // clipped by the store; lines past N and warps whose 32 queries all lie
    // past N skip it).
    uint8_t* const ostg = smem + OFF_OST + sw * OST_BYTES;
    auto finish_unit = [&](int ui, int clast, float l) -> bool {
      if (!warp_wait_or_abort(&bars->p_free[r][clast & 1], (clast >> 1) & 1, ab)) return false;
      tc::tc_fence_after();
      uint32_t ov[32];
      tc::tmem_ld32(tb + TM_O, ov);
      tc::tmem_ld_wait();
      // O is in registers: its columns may take the next unit's sums.
      tc::tc_fence_before();
      tc::mbar_arrive(&bars->o_free[r]);
      const Unit fu = decode_unit(p.unit0 + blockIdx.x + ui * gridDim.x, p);
      const int fi = fu.rg * R + r, fj = fu.j0 + (warp & 3) * 32;
      if (fi < N && fj < N) {
        // A query row has l in [2^-16, 2^100) unless its logits left that range
        // (a uniform row or query has l = its count of real keys): those rows
        // are recomputed exactly.
        const bool exact = fj + lane < N && !(l >= 0x1p-16f && l < 0x1p100f);
        const float inv = __fdividef(1.0f, l);   // l lies in [2^-16, 2^100): the fast form is exact enough
        uint32_t po[16];
#pragma unroll
        for (int e = 0; e < DH; e += 2)
          po[e / 2] = tc::pack_bf16x2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
        // The previous store (if any) has read the staging tile.
        if (lane == 0) tc::tma_store_wait_read<0>();
        __syncwarp();
        if (__builtin_expect(exact, 0)) {
          const long long base = (long long)fu.b * p.sb + (long long)fi * p.sl + fu.t * DH;
          const long long plane = ((long long)fu.b * p.h + fu.t) * N * N;
          const int a = fj + lane;             // the query's position along the line
          exact_row(p.q + base + (long long)a * p.sx, p.k + base, p.v + base, p.sx,
                    p.bias32 + plane + (p.ending ? (long long)a : (long long)a * N),
                    p.ending ? (long long)N : 1ll,
                    p.mask_mode == TRI_ATTN_MASK_QUERY_KEY
                        ? nullptr
                        : p.mbits + ((long long)fu.b * N + fi) * p.words,
                    N, ostg, lane);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *(uint4*)(ostg + tc::swz_offset(lane, q, 64)) =
                make_uint4(po[4 * q], po[4 * q + 1], po[4 * q + 2], po[4 * q + 3]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_store_4d(&map_o, ostg, fu.t * DH, fj, fi, fu.b);
          tc::tma_store_commit();
        }
      }
      return true;
    };
    bool ok = true;
    SoftIt its{0, 0, 0, 0};                         // this warp's sub-tile stream
    float l_prev = 0.f;
    for (int ui = 0; ok && ui < my_units; ++ui) {
      const bool uni = nx_any == 0u;
      const uint32_t* mrow = nx_mrow;
      if (ui + 1 < my_units)
        unit_loads(decode_unit(p.unit0 + blockIdx.x + (ui + 1) * gridDim.x, p), nx_any, nx_mrow);
      float l_run = 0.f;
      // Warp-uniform unit state: whether any lane has a key-keeping query row,
      // and whether every lane has one.
      const bool unit_live = __any_sync(0xffffffffu, !uni);
      const bool all_live = __all_sync(0xffffffffu, !uni);
      uint2 nbits = __ldg((const uint2*)mrow);
      for (int kt = 0; ok && kt < KT; ++kt, advance(its, KT)) {
        const int c = its.c;
        const uint2 mb = nbits;
        if (kt + 1 < KT) nbits = __ldg((const uint2*)(mrow + 2 * (kt + 1)));
        const int left = N - kt * BK;
        const uint32_t rl0 = real_bits(left, 0), rl1 = real_bits(left, 1);
        // Keys kept by this lane (query-key: its own query row; row-key: the
        // line, the same for the whole warp).
        const uint32_t kb0 = rl0 & mb.x, kb1 = rl1 & mb.y;
        // Row-key: S of a dropped key is set to -inf. Query-key: the bias plane
        // already holds -inf there.
        const uint32_t bw0 = qk_mode ? rl0 : kb0, bw1 = qk_mode ? rl1 : kb1;
        const bool all_kept = (bw0 & bw1) == 0xffffffffu;      // warp-uniform
        const bool tile_keys = (bw0 | bw1) != 0u;              // warp-uniform
        const bool live = !uni && tile_keys;
        const uint32_t brow = brow0 + its.bs * BIAS_BYTES;
        // The bias stage and S(c): both barriers are polled back to back so
        // that their latencies overlap, then one vote settles them.
        bool okk = tc::mbar_try_wait(&bars->b_full[its.bs], its.bph);
        bool oks = tc::mbar_try_wait(&bars->s_ready[r][c & 1], (c >> 1) & 1);
        if (!okk) okk = wait_or_abort_slow(&bars->b_full[its.bs], its.bph, ab);
        if (okk && !oks) oks = wait_or_abort_slow(&bars->s_ready[r][c & 1], (c >> 1) & 1, ab);
        if (!__all_sync(0xffffffffu, okk && oks)) { ok = false; break; }
        const bool any_live = unit_live && tile_keys;
        tc::tc_fence_after();
        const uint32_t tsb = tb + (c & 1) * TM_S1;     // S(c), then P(c) over it
        float2 x2[BK / 2];
        uint4 bh0[4], bh1[4];
        float tsum = 0.f;
        if (any_live) {
          tc::tmem_ld32(tsb, *(uint32_t(*)[32])&x2[0]);
          tc::tmem_ld32(tsb + 32, *(uint32_t(*)[32])&x2[16]);
          load_bias_half(brow, 0, bh0);
          load_bias_half(brow, 1, bh1);
          tc::tmem_ld_wait();
          if (!all_kept) {
            // Dropped keys: S = -inf, which the bias add keeps at -inf (P = 0).
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              if (!((bw0 >> (2 * k)) & 1u)) x2[k].x = -INFINITY;
              if (!((bw0 >> (2 * k + 1)) & 1u)) x2[k].y = -INFINITY;
              if (!((bw1 >> (2 * k)) & 1u)) x2[16 + k].x = -INFINITY;
              if (!((bw1 >> (2 * k + 1)) & 1u)) x2[16 + k].y = -INFINITY;
            }
          }
          uint32_t pk[16];
          float2 ts2;
          if (all_live) {
            ts2 = p_half_fast(x2, bh0, 0, pk);
            tc::tmem_st16(tsb, pk);
            ts2 = __fadd2_rn(ts2, p_half_fast(x2, bh1, 1, pk));
            tc::tmem_st16(tsb + 16, pk);
          } else {
            const uint32_t w0 = uni ? rl0 : 0u, w1 = uni ? rl1 : 0u;
            ts2 = p_half(x2, bh0, 0, 0.f, live, w0, pk);
            tc::tmem_st16(tsb, pk);
            ts2 = __fadd2_rn(ts2, p_half(x2, bh1, 1, 0.f, live, w1, pk));
            tc::tmem_st16(tsb + 16, pk);
          }
          tsum = ts2.x + ts2.y;
        } else {
          // No lane of the warp keeps a key of this sub-tile: P is 1 on the real
          // keys of a uniform row or query, else 0.
          uint32_t pk[16];
          p_half_const(uni ? rl0 : 0u, pk);
          tc::tmem_st16(tsb, pk);
          p_half_const(uni ? rl1 : 0u, pk);
          tc::tmem_st16(tsb + 16, pk);
        }
        // The bias stage is read: release it.
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars->b_empty[its.bs]);
        if (live) {
          l_run += tsum;
        } else if (uni) {
          l_run += (float)(__popc(rl0) + __popc(rl1));
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(&bars->p_full[r][c & 1]);
        if (kt == 0 && ui >= 1) {
          // The previous unit's epilogue, after this unit's first sub-tile.
          if (!finish_unit(ui - 1, c - 1, l_prev)) { ok = false; break; }
        }
      }
      if (!ok) break;
      l_prev = l_run;
    }
    if (ok && my_units > 0) finish_unit(my_units - 1, my_units * KT - 1, l_prev);
    if (lane == 0) tc::tma_store_wait_all<0>();
  }

  // ---------------- teardown
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    for (int ui = q_issued - 1; ui >= 0 && ui >= q_issued - 2; --ui)
      drain_wait(&bars->q_full[ui & 1], (ui >> 1) & 1);
    for (int g = kv_issued - 1; g >= 0 && g >= kv_issued - KV_STAGES; --g)
      drain_wait(&bars->kv_full[g % KV_STAGES], (g / KV_STAGES) & 1);
    for (int g = b_issued - 1; g >= 0 && g >= b_issued - B_STAGES; --g)
      drain_wait(&bars->b_full[g % B_STAGES], (g / B_STAGES) & 1);
  }
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
#undef ab
}

// The attention's bias plane from K1's cell-order plane C (fp32, log2(e) *
// bias, -inf where the query-key reading drops the key): row (b, t, query a)
// holds the biases of the keys along line a, which is row a of C (starting
// node) or column a (ending node: the bias of key k for query a is that of
// cell (k, a)). Each row is stored in fp16 minus its largest entry: the softmax
// over keys is unchanged by a per-row constant, and the entries that carry the
// weight (near the row's largest) are then small in magnitude, where fp16 is
// precise. A block takes 8 rows of one (b, t) plane, one warp per row, and
// walks the keys 128 at a time (4 per lane), once for the row maximum and once
// to write; for the ending node each step first moves a 128-key x 8-query
// block of C (32 contiguous bytes per key) through shared memory. A row with
// every key dropped stays -inf.
__global__ void __launch_bounds__(256)
bias_rows(const float* __restrict__ C, int N, int Nb, int ending, __half* __restrict__ P) {
  __shared__ float tile[8][132];
  const int a0 = blockIdx.x * 8;
  const long long plane = blockIdx.y;
  const float* Cp = C + plane * N * N;
  __half* Pp = P + plane * N * Nb;
  const int wq = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = a0 + wq;                          // this warp's row
  float m = -INFINITY;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll 1
    for (int k0 = 0; k0 < N; k0 += 128) {
      float v[4];
      if (ending) {
        // Thread i moves C[k0 + i / 2][a0 + 4 (i & 1) .. + 3] to tile[query][key].
        const int kk = k0 + (threadIdx.x >> 1), qa = 4 * (threadIdx.x & 1);
        __syncthreads();                          // the previous step has read the tile
#pragma unroll
        for (int e = 0; e < 4; ++e)
          tile[qa + e][threadIdx.x >> 1] =
              (kk < N && a0 + qa + e < N) ? Cp[(long long)kk * N + a0 + qa + e] : -INFINITY;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = tile[wq][4 * lane + e];
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = k0 + 4 * lane + e;
          v[e] = (k < N && a < N) ? Cp[(long long)a * N + k] : -INFINITY;
        }
      }
      if (pass == 0) {
        m = fmaxf(fmaxf(m, fmaxf(v[0], v[1])), fmaxf(v[2], v[3]));
      } else if (a < N) {
        const int k = k0 + 4 * lane;
        __half hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) hv[e] = __float2half_rn(m == -INFINITY ? -INFINITY : v[e] - m);
        if (k + 3 < N) {                          // 8-byte store: Nb and k are multiples of 4
          *(uint2*)(Pp + (long long)a * Nb + k) = *(const uint2*)hv;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (k + e < N) Pp[(long long)a * Nb + k + e] = hv[e];
        }
      }
    }
    if (pass == 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
  }
}

// One warp per mask row (b, r): bit k of word k/32 is pair_mask[b, r, k] != 0
// for k < N (0 beyond, up to `words` words), and any[row] says whether the row
// keeps some key.
__global__ void mask_summary(const int32_t* __restrict__ mask, int N, long long rows, int words,
                             uint32_t* __restrict__ bits, unsigned char* __restrict__ any) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  unsigned found = 0;
  for (int wd = 0; wd < words; ++wd) {
    const int k = wd * 32 + lane;
    const bool keep = k < N && mask[row * N + k] != 0;
    const unsigned w = __ballot_sync(0xffffffffu, keep);
    found |= w;
    if (lane == 0) bits[row * words + wd] = w;
  }
  if (lane == 0) any[row] = found != 0;
}

// Ending node: line (b, a) is column a of the mask (key k = grid row k). A
// block takes 32 columns of one batch, lane = column a; warp wp forms the
// words w = wp, wp + 8, ... (bit kk of word w: pair_mask[b, 32 w + kk, a] != 0,
// each of its 32 loads one coalesced 128-byte row segment across the warp),
// and the block ORs them into the column's "keeps some key" flag.
__global__ void __launch_bounds__(256)
mask_summary_cols(const int32_t* __restrict__ mask, int N, int words, uint32_t* __restrict__ bits,
                  unsigned char* __restrict__ any) {
  __shared__ uint32_t found[8][32];
  const int cblocks = (N + 31) >> 5;
  const long long b = blockIdx.x / cblocks;
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int a = (int)(blockIdx.x % cblocks) * 32 + lane;
  uint32_t acc = 0;
  if (a < N) {
    const int32_t* col = mask + b * N * N + a;
    for (int w = wp; w < words; w += 8) {
      uint32_t word = 0;
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const int k = 32 * w + kk;
        if (k < N && col[(long long)k * N] != 0) word |= 1u << kk;
      }
      bits[(b * N + a) * words + w] = word;
      acc |= word;
    }
  }
  found[wp][lane] = acc;
  __syncthreads();
  if (wp == 0 && a < N) {
#pragma unroll
    for (int i = 1; i < 8; ++i) acc |= found[i][lane];
    any[b * N + a] = acc != 0;
  }
}
}  // namespace k2


// ---------------------------------------------------------------------------
// K3: gate multiply (prologue) + output projection
// ---------------------------------------------------------------------------
namespace k3 {
constexpr int BM = 128;
constexpr int KD = 128;
// Warps 0-3 form g * o (one cell row per thread), warps 4-7 drain the
// accumulator (TMEM lane quarter = warp % 4), warp 8 TMA, warp 9 MMA: the gate
// product of tile t + 1 is formed while the epilogue drains tile t.
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr uint32_t T_BYTES = BM * KD * 2;           // 32 KB tile (two K-halves)
constexpr uint32_t OFF_W = 0;                       // Wo, 32 KB
constexpr uint32_t OFF_G = OFF_W + T_BYTES;         // g tiles [2]; become the A operand
constexpr uint32_t OFF_O = OFF_G + 2 * T_BYTES;     // o tiles [2]
// Output staging: per epilogue warp two 32-row x 32-channel bf16 tiles (64-byte
// rows, 64-byte swizzle), each written by one TMA store.
constexpr uint32_t STG_BYTES = 32 * 64;
constexpr uint32_t OFF_STG = OFF_O + 2 * T_BYTES;   // [4 warps][2]
constexpr uint32_t OFF_BO = OFF_STG + 4 * 2 * STG_BYTES;   // bo fp32 [128]
constexpr uint32_t OFF_BAR = OFF_BO + KD * 4;
constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;

struct Bars {
  uint64_t w_full, in_full[2], in_empty[2], a_ready[2], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort;
};

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

// TMA coordinates (x, y, z) of tile `tile` after the channel coordinate.
struct TileAt { int x, y, z; };
__device__ __forceinline__ TileAt tile_at(const Params& p, int tile) {
  if (!p.cols) return {tile * BM, 0, 0};
  const int line = tile / p.tpl;
  return {(tile - line * p.tpl) * BM, line % p.N, line / p.N};
}

__global__ void __launch_bounds__(kThreads, 1)
gate_out_tc(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_o,
            const __grid_constant__ CUtensorMap map_wo, const __grid_constant__ CUtensorMap map_out,
            const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = (Bars*)(smem + OFF_BAR);
  float* s_bo = (float*)(smem + OFF_BO);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Abort ab{&bars->abort, p.dev_err, p.polls};
  if (tid == 0) {
    tc::mbar_init(&bars->w_full, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars->in_full[b], 1);
      tc::mbar_init(&bars->in_empty[b], 1);
      tc::mbar_init(&bars->a_ready[b], 128);
      tc::mbar_init(&bars->acc_full[b], 1);
      tc::mbar_init(&bars->acc_empty[b], 128);
    }
    tc::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  for (int i = tid; i < KD; i += kThreads) s_bo[i] = p.bo[i];
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&bars->tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int my_tiles = 0;
  for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) ++my_tiles;
  int issued = 0;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&map_g);
      tc::tma_prefetch_desc(&map_o);
      tc::tma_prefetch_desc(&map_wo);
      tc::mbar_arrive_expect_tx(&bars->w_full, T_BYTES);
      tc::tma_load_2d(smem + OFF_W, &map_wo, &bars->w_full, 0, 0);
      tc::tma_load_2d(smem + OFF_W + 16384, &map_wo, &bars->w_full, 64, 0);
      for (int it = 0; it < my_tiles; ++it) {
        const int b = it & 1;
        if (it >= 2 && !wait_or_abort(&bars->in_empty[b], ((it >> 1) - 1) & 1, ab)) break;
        const TileAt at = tile_at(p, p.tile0 + blockIdx.x + it * gridDim.x);
        uint8_t* gs = smem + OFF_G + b * T_BYTES;
        uint8_t* os = smem + OFF_O + b * T_BYTES;
        tc::mbar_arrive_expect_tx(&bars->in_full[b], 2 * T_BYTES);
        tc::tma_load_4d(gs, &map_g, &bars->in_full[b], 0, at.x, at.y, at.z);
        tc::tma_load_4d(gs + 16384, &map_g, &bars->in_full[b], 64, at.x, at.y, at.z);
        tc::tma_load_4d(os, &map_o, &bars->in_full[b], 0, at.x, at.y, at.z);
        tc::tma_load_4d(os + 16384, &map_o, &bars->in_full[b], 64, at.x, at.y, at.z);
        issued = it + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t w0 = tc::smem_addr(smem + OFF_W);
      bool ok = wait_or_abort(&bars->w_full, 0, ab);
      for (int it = 0; ok && it < my_tiles; ++it) {
        const int b = it & 1;
        if (!wait_or_abort(&bars->a_ready[b], (it >> 1) & 1, ab)) break;
        if (it >= 2 && !wait_or_abort(&bars->acc_empty[b], ((it >> 1) - 1) & 1, ab)) break;
        tc::tc_fence_after();
        const uint32_t a0 = tc::smem_addr(smem + OFF_G + b * T_BYTES);
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t ko = (ks >> 2) * 16384 + (ks & 3) * 32;
          tc::mma_bf16_ss(tmem + b * 128, tc::smem_desc(a0 + ko, 16, 1024, tc::SWZ_128B),
                          tc::smem_desc(w0 + ko, 16, 1024, tc::SWZ_128B), idesc, ks > 0);
        }
        tc::mma_commit(&bars->acc_full[b]);
        tc::mma_commit(&bars->in_empty[b]);
      }
      tc::mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0);
    }
  } else if (warp < 4) {
    // ---------------- gate: a = g * o in place (one cell row per thread)
    const int r = tid;
    for (int it = 0; it < my_tiles; ++it) {
      const int b = it & 1;
      if (!warp_wait_or_abort(&bars->in_full[b], (it >> 1) & 1, ab)) break;
      uint8_t* gs = smem + OFF_G + b * T_BYTES;
      const uint8_t* os = smem + OFF_O + b * T_BYTES;
#pragma unroll 4
      for (int c = 0; c < 16; ++c) {
        const uint32_t off = (c >> 3) * 16384 + tc::swz_offset(r, c & 7, 128);
        const uint4 gu = *(const uint4*)(gs + off);
        const uint4 ou = *(const uint4*)(os + off);
        // bf16 x bf16 is exact in fp32, so the packed bf16 product rounds it once.
        const uint32_t ga[4] = {gu.x, gu.y, gu.z, gu.w}, oa[4] = {ou.x, ou.y, ou.z, ou.w};
        uint32_t res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 pr = __hmul2(*(const __nv_bfloat162*)&ga[e], *(const __nv_bfloat162*)&oa[e]);
          res[e] = *(const uint32_t*)&pr;
        }
        *(uint4*)(gs + off) = make_uint4(res[0], res[1], res[2], res[3]);
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars->a_ready[b]);
    }
  } else if (warp < 8) {
    // ---------------- epilogue: cell row = TMEM lane of this warp's quarter;
    // each 32-row x 32-channel chunk leaves through a swizzled staging tile and
    // one TMA store (rows past the last cell, or past the end of a column, are
    // clipped by the tensor bounds).
    const int q4 = warp & 3;
    uint8_t* const stg0 = smem + OFF_STG + q4 * 2 * STG_BYTES;
    int nst = 0;                                  // TMA stores issued by this warp
    for (int it = 0; it < my_tiles; ++it) {
      const int b = it & 1;
      if (!warp_wait_or_abort(&bars->acc_full[b], (it >> 1) & 1, ab)) break;
      tc::tc_fence_after();
      const TileAt at = tile_at(p, p.tile0 + blockIdx.x + it * gridDim.x);
      // Chunk ch + 1 is loaded from TMEM while chunk ch is converted and stored.
      uint32_t accb[2][32];
      tc::tmem_ld32(tc::tmem_addr(tmem, q4 * 32, b * 128), accb[0]);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        tc::tmem_ld_wait();
        if (ch + 1 < 4) tc::tmem_ld32(tc::tmem_addr(tmem, q4 * 32, b * 128 + (ch + 1) * 32), accb[(ch + 1) & 1]);
        const uint32_t (&acc)[32] = accb[ch & 1];
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = tc::pack_bf16x2(__uint_as_float(acc[2 * e]) + s_bo[ch * 32 + 2 * e],
                                  __uint_as_float(acc[2 * e + 1]) + s_bo[ch * 32 + 2 * e + 1]);
        uint8_t* stg = stg0 + (nst & 1) * STG_BYTES;
        if (nst >= 2) {                           // the store two back has read this tile
          if (lane == 0) tc::tma_store_wait_read<1>();
          __syncwarp();
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *(uint4*)(stg + tc::swz_offset(lane, e, 64)) =
              make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::tma_store_4d(&map_out, stg, ch * 32, at.x + q4 * 32, at.y, at.z);
          tc::tma_store_commit();
        }
        ++nst;
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&bars->acc_empty[b]);
    }
    if (lane == 0) tc::tma_store_wait_all<0>();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kTmaWarp && lane == 0) {
    drain_wait(&bars->w_full, 0);
    for (int it = issued - 1; it >= 0 && it >= issued - 2; --it)
      drain_wait(&bars->in_full[it & 1], (it >> 1) & 1);
  }
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 256);
}
}  // namespace k3

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
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

bool map_rows_bf16(CUtensorMap* m, const void* base, long long rows, int box_rows) {
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// A (B, N, N, 128) bf16 activation seen as (channel, position x along a line,
// line a, batch b): lines are the grid's rows (starting node: cell (a, x)) or
// its columns (ending node: cell (x, a)). Box: one head (32 channels) x box_x
// positions of one line.
bool map_lines(CUtensorMap* m, const void* base, int B, int N, int box_x, bool ending) {
  const cuuint64_t cell = 256, row = (cuuint64_t)N * 256;
  cuuint64_t dims[4] = {128, (cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {ending ? row : cell, ending ? cell : row, (cuuint64_t)N * row};
  cuuint32_t box[4] = {32, (cuuint32_t)box_x, 1, 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_64B);
}

// K3's view of a (B, N, N, 128) bf16 activation as (channel, x, y, z): in cell
// order (x = cell, y = z = 0) or by columns (x = grid row i, y = column j,
// z = batch b). Box: box_ch channels x box_x positions along x.
bool map_k3(CUtensorMap* m, const void* base, const tri_attn_s* t, bool cols, int box_ch,
            int box_x, CUtensorMapSwizzle swz) {
  const cuuint64_t cell = 256, row = (cuuint64_t)t->N * 256, cells = (cuuint64_t)t->cells;
  const cuuint64_t dims_flat[4] = {128, cells, 1, 1}, strides_flat[3] = {cell, cell * cells,
                                                                         cell * cells};
  const cuuint64_t dims_cols[4] = {128, (cuuint64_t)t->N, (cuuint64_t)t->N, (cuuint64_t)t->B};
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
  k1::Consts consts;                        // LayerNorm / gate-bias / pair-bias weights (fp32)
  CUtensorMap map_w, map_q, map_k, map_v, map_b, map_wo;
  CUtensorMap map_g, map_o;                // K3 loads, cell-order tiles
  CUtensorMap map_gc, map_oc;              // K3 loads, column tiles
  CUtensorMap st_q, st_k, st_v, st_g;      // K1 output stores: (cells, 128) bf16, 32 x 32 boxes
  CUtensorMap map_os;                      // K2 output stores: one head x 32 queries of a row
  float* bias32;             // (B, h, N, N) fp32 pair bias in cell order (K1's output)
  unsigned char* row_any;    // (B*N) mask rows keeping some key
  uint32_t* mbits;           // (B*N, words) mask bits
  int words;
  int num_sms;
  int Nb;
  // Host-buffer pipeline (created at its first use): copy streams and events.
  cudaStream_t copy_in, copy_out;
  cudaEvent_t ev[kHostEvents];
};

int round_up(int a, int b) { return (a + b - 1) / b * b; }


}  // namespace

bool tri_tc_supported(int B, int N, int D, int h) {
  const long long cells = (long long)B * N * N;
  return D == 128 && h == 4 && N >= 1 && N <= 8192 && cells < (1ll << 31) &&
         (long long)B * N < (1ll << 31) / 8;
}

size_t tri_tc_extra_bytes(int B, int N, int, int h) {
  // the attention's fp16 bias plane (rows padded to Nb) beside K1's fp32 one;
  // plus the mask summary
  const size_t Nb = (size_t)round_up(N, 8);
  return (size_t)B * h * N * Nb * 2 + (size_t)B * N + (size_t)B * N * 2 * ((N + 63) / 64) * 4 +
         512;
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
  if (e == cudaSuccess) e = cudaMalloc((void**)&st->row_any, (size_t)B * N);
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
  if (e == cudaSuccess) e = cudaMemcpyAsync(st->consts.gw, t->wb_f32, (size_t)h * D * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
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

  const long long cells = t->cells;
  bool ok = map_rows_bf16(&st->map_w, t->w_proj, 512, 256);
  ok = ok && map_lines(&st->map_q, t->q, B, N, k2::BQ, t->ending);
  ok = ok && map_lines(&st->map_k, t->k, B, N, k2::KVK, t->ending);
  ok = ok && map_lines(&st->map_v, t->v, B, N, k2::KVK, t->ending);
  ok = ok && map_lines(&st->map_os, t->o, B, N, 32, t->ending);
  {
    cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)B * h};
    cuuint64_t strides[2] = {(cuuint64_t)st->Nb * 2, (cuuint64_t)N * st->Nb * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)k2::BQ, 1};   // 128-byte rows for SWIZZLE_128B
    ok = ok && make_map(&st->map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, t->bias, dims, strides,
                        box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  ok = ok && map_k3(&st->map_g, t->g, t, false, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map_k3(&st->map_gc, t->g, t, true, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  {
    void* outs[4] = {t->q, t->k, t->v, t->g};
    CUtensorMap* maps[4] = {&st->st_q, &st->st_k, &st->st_v, &st->st_g};
    for (int m = 0; m < 4 && ok; ++m) {
      cuuint64_t dims[2] = {128, (cuuint64_t)cells};
      cuuint64_t strides[1] = {256};
      cuuint32_t box[2] = {32, 32};
      ok = make_map(maps[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, outs[m], dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_64B);
    }
  }
  ok = ok && map_k3(&st->map_o, t->o, t, false, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map_k3(&st->map_oc, t->o, t, true, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map_rows_bf16(&st->map_wo, t->w_out, 128, 128);
  if (!ok) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(k1::ln_proj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, k1::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k2::row_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, k2::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k3::gate_out_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, k3::SMEM);
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
  p1.q = (__nv_bfloat16*)t->q; p1.k = (__nv_bfloat16*)t->k; p1.v = (__nv_bfloat16*)t->v;
  p1.g = (__nv_bfloat16*)t->g; p1.bias32 = st->bias32; p1.dev_err = t->dev_err;
  p1.polls = t->wait_limit;
  p1.q_scale = kLog2e / sqrtf((float)t->d);
  const int grid = n < st->num_sms ? n : st->num_sms;
  k1::ln_proj_tc<<<grid, k1::kThreads, k1::SMEM, s>>>(map_x, st->map_w, st->st_q, st->st_k,
                                                      st->st_v, st->st_g, p1, st->consts);
  return cudaGetLastError();
}

// The mask summary of every line.
cudaError_t launch_mask(tri_attn_s* t, cudaStream_t s, const int32_t* mask, int& mark) {
  TcState* st = (TcState*)t->tc;
  const int B = t->B, N = t->N;
  const long long rows = (long long)B * N;
  if (!t->ending) {
    k2::mask_summary<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(mask, N, rows, st->words,
                                                              st->mbits, st->row_any);
    tri_mark(t, s, mark++, "mask_summary");
  } else {
    const unsigned blocks = (unsigned)(B * (long long)((N + 31) / 32));
    k2::mask_summary_cols<<<blocks, 256, 0, s>>>(mask, N, st->words, st->mbits, st->row_any);
    tri_mark(t, s, mark++, "mask_summary_cols");
  }
  return cudaGetLastError();
}

// The attention's bias plane from K1's (after every K1 tile).
cudaError_t launch_bias_rows(tri_attn_s* t, cudaStream_t s, int& mark) {
  TcState* st = (TcState*)t->tc;
  const dim3 grid((unsigned)((t->N + 7) / 8), (unsigned)(t->B * t->h));
  k2::bias_rows<<<grid, 256, 0, s>>>(st->bias32, t->N, st->Nb, t->ending ? 1 : 0,
                                      (__half*)t->bias);
  tri_mark(t, s, mark++, "bias_rows");
  return cudaGetLastError();
}

// K2's work units are (b, row group, head, query tile), query tile fastest.
int k2_row_groups(const tri_attn_s* t) { return (t->N + k2::R - 1) / k2::R; }
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
  p2.mbits = st->mbits; p2.row_any = st->row_any;
  p2.dev_err = t->dev_err;
  p2.polls = t->wait_limit;
  p2.q = (const __nv_bfloat16*)t->q;
  p2.k = (const __nv_bfloat16*)t->k;
  p2.v = (const __nv_bfloat16*)t->v;
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
  k2::row_attn_tc<<<g2, k2::kThreads, k2::SMEM, s>>>(st->map_q, st->map_k, st->map_v, st->map_b,
                                                      st->map_os, p2);
  return cudaGetLastError();
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
  k3::gate_out_tc<<<grid, k3::kThreads, k3::SMEM, s>>>(cols ? st->map_gc : st->map_g,
                                                       cols ? st->map_oc : st->map_o,
                                                       st->map_wo, map_out, p3);
  return cudaGetLastError();
}

}  // namespace

cudaError_t tri_tc_forward(tri_attn_s* t, cudaStream_t s, const void* x, const int32_t* mask,
                           void* out) {
  const int ntiles = num_tiles(t);
  CUtensorMap map_x, map_out;
  if (!map_rows_bf16(&map_x, x, t->cells, 128) || !map_out_k3(&map_out, out, t, false))
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
  if (!map_rows_bf16(&map_x, dx, t->cells, 128) || !map_out_k3(&map_out, dout, t, cols))
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
    return (long long)(g / rgs) * t->N + std::min((g % rgs) * k2::R, t->N);
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
