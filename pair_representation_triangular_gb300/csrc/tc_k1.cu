// K1 of the bf16 tensor-core path: LayerNorm as the prologue of one
// concatenated projection GEMM, x_hat [128 cells x D] . [Wq|Wk|Wv|Wg]^T -> 4D
// TMEM columns; the epilogue writes q (times log2(e)/sqrt(d)) and k in bf16,
// v in fp16 (times a power of 2, folded into the packed Wv rows, that keeps it
// in range; the attention's P V runs on fp16 operands) and sigmoid(g + bg) in
// bf16. The h pair-bias outputs (Wb x_hat, with gamma and
// beta folded into Wb) come out of the LayerNorm's statistics pass on the CUDA
// cores and go, scaled by log2(e), to an fp32 plane in cell order.
//
// Passages followed: POPCORNBENCH "Kimi-K2.6 l2_p6", forward op list steps
// 1-9 (LayerNorm, the q/k/v/gate/bias projections, the gate sigmoid) and the
// layer definitions (which projections carry a bias).
#include "tc_device.cuh"
#include "tc_kernels.cuh"

namespace tri_tc {
namespace k1 {

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

// Persistent: CTA c serves 128-cell tiles c, c + G, ... [Wq;Wk;Wv;Wg] (bf16,
// K-major, 8 D^2 bytes) stays in shared memory. Per tile the x tile arrives by
// TMA; the 256 workers normalise it in place (the two threads of a cell each
// own one half of its channels; each takes the row statistics and up to
// ceil(h/2) of the h bias outputs from the whole row in one shifted pass, the
// bias through gamma and beta folded into Wb); the MMA warp issues the two
// N = 2D halves (q|k, v|g) into TMEM columns 0 .. 2D-1 and 2D .. 4D-1, each with
// its own full/empty barriers, so the next tile's first half can start while
// the epilogue still reads the second. Warps 0-7 LayerNorm (warp q takes
// channel half 0 of rows 32q..32q+31, warp q + 4 half 1), warps 8-15 epilogue
// (two per TMEM lane quarter), warp 16 TMA, warp 17 MMA.
template <int D, int H>
__global__ void __launch_bounds__(kThreads, 1)
ln_proj_tc(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
           const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
           const Params p, const __grid_constant__ Consts cst) {
  using S = Shape<D>;
  constexpr int XSW = S::XSW, CH16 = S::CH16;
  constexpr int HPT = (H + 1) / 2;         // bias heads per thread of a row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = (Bars*)(smem + S::OFF_BAR);
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
    tc::tmem_alloc(&bars->tmem_base, S::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int my_tiles = 0;
  for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) ++my_tiles;
  int issued = 0;                          // tile loads issued (producer thread)
  pdl_trigger();
  // x, the mask and every output may belong to the previous kernel on the
  // stream; only the resident weights are loaded before its completion.
  if (warp != kTmaWarp) pdl_wait();

  if (warp == kTmaWarp) {
    // ---------------- TMA producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&map_x);
      tc::tma_prefetch_desc(&map_w);
      tc::mbar_arrive_expect_tx(&bars->w_full, S::W_BYTES);
      for (int kh = 0; kh < S::KH; ++kh)
        for (int nh = 0; nh < 2; ++nh)
          tc::tma_load_2d(smem + S::OFF_W + kh * S::W_HALF + nh * S::NHALF * XSW, &map_w,
                          &bars->w_full, kh * S::HC, nh * S::NHALF);
      pdl_wait();
      for (int it = 0; it < my_tiles; ++it) {
        const int b = it & 1;
        if (it >= 2 && !wait_or_abort(&bars->x_empty[b], ((it >> 1) - 1) & 1, ab)) break;
        const int tile = p.tile0 + blockIdx.x + it * gridDim.x;
        uint8_t* xs = smem + S::OFF_X + b * S::X_BYTES;
        tc::mbar_arrive_expect_tx(&bars->x_full[b], S::X_BYTES);
        for (int kh = 0; kh < S::KH; ++kh)
          tc::tma_load_2d(xs + kh * S::X_HALF, &map_x, &bars->x_full[b], kh * S::HC, tile * BM);
        issued = it + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, S::NHALF, 0, 0);
      constexpr uint32_t swm = swz_mode(XSW);
      const uint32_t w0 = tc::smem_addr(smem + S::OFF_W);
      bool ok = wait_or_abort(&bars->w_full, 0, ab);
      for (int it = 0; ok && it < my_tiles; ++it) {
        const int b = it & 1;
        if (!wait_or_abort(&bars->a_ready[b], (it >> 1) & 1, ab)) break;
        const uint32_t a0 = tc::smem_addr(smem + S::OFF_X + b * S::X_BYTES);
        for (int nh = 0; nh < 2 && ok; ++nh) {
          if (it >= 1 && !wait_or_abort(&bars->acc_empty[nh], (it - 1) & 1, ab)) { ok = false; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t kh = ks / S::KSTEPS_PER_HALF, kin = ks % S::KSTEPS_PER_HALF;
            const uint64_t ad = tc::smem_desc(a0 + kh * S::X_HALF + kin * 32, 16, 8 * XSW, swm);
            const uint64_t bd = tc::smem_desc(w0 + kh * S::W_HALF + nh * S::NHALF * XSW + kin * 32,
                                              16, 8 * XSW, swm);
            tc::mma_ss(tmem + nh * S::NHALF, ad, bd, idesc, ks > 0);
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
    // Parameter pairs (one 8-byte constant load each): this thread's bias heads
    // and the LayerNorm affine.
    const float2* gw2[HPT];
#pragma unroll
    for (int t2 = 0; t2 < HPT; ++t2) gw2[t2] = (const float2*)cst.gw[hh * HPT + t2];
    const float2* gamma2 = (const float2*)cst.gamma;
    const float2* beta2 = (const float2*)cst.beta;
    const long long NN = (long long)p.N * p.N;
    bool ok = true;
    for (int it = 0; ok && it < my_tiles; ++it) {
      const int b = it & 1;
      if (!warp_wait_or_abort(&bars->x_full[b], (it >> 1) & 1, ab)) { ok = false; break; }
      const int tile = p.tile0 + blockIdx.x + it * gridDim.x;
      const long long cell = (long long)tile * BM + r;
      uint8_t* xs = smem + S::OFF_X + b * S::X_BYTES;
      auto chunk_at = [&](int c) -> uint8_t* {
        return xs + (c / CH16) * S::X_HALF + swz(r, c % CH16, XSW);
      };
      // One pass over the whole row, shifted by its first channel K so that the
      // sums do not cancel: the row statistics and this thread's bias heads
      // (hh * HPT ..) through the folded constants of k1::Consts.
      const float K0 = bf16_lo(((const uint4*)chunk_at(0))->x);
      const float2 nk2 = make_float2(-K0, -K0);
      float2 s2 = make_float2(0.f, 0.f), q2 = make_float2(0.f, 0.f);
      float2 bp[HPT];
#pragma unroll
      for (int t2 = 0; t2 < HPT; ++t2) bp[t2] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 u = *(const uint4*)chunk_at(c);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i0 = c * 8 + 2 * e;
          const float2 d = __fadd2_rn(make_float2(bf16_lo(w4[e]), bf16_hi(w4[e])), nk2);
          s2 = __fadd2_rn(s2, d);
          q2 = __ffma2_rn(d, d, q2);
#pragma unroll
          for (int t2 = 0; t2 < HPT; ++t2)
            bp[t2] = __ffma2_rn(d, gw2[t2][i0 / 2], bp[t2]);
        }
      }
      const float S1 = (s2.x + s2.y) * (1.0f / D);             // mean of x - K
      const float var = fmaxf((q2.x + q2.y) * (1.0f / D) - S1 * S1, 0.f);
      const float mean = K0 + S1;
      const float rstd = rsqrtf(var + 1e-5f);
      float bsum[HPT];
#pragma unroll
      for (int t2 = 0; t2 < HPT; ++t2)
        bsum[t2] = rstd * ((bp[t2].x + bp[t2].y) - S1 * cst.gws[hh * HPT + t2]) + cst.bw[hh * HPT + t2];
      // Normalise this thread's half of the channels, rounded to bf16 as the MMA
      // sees it.
      constexpr int MYC = D / 16;                              // chunks per thread
      const float2 rs2 = make_float2(rstd, rstd), nm2 = make_float2(-mean * rstd, -mean * rstd);
      uint32_t mine[4 * MYC];
#pragma unroll
      for (int c = 0; c < MYC; ++c) {
        const uint4 u = *(const uint4*)chunk_at(hh * MYC + c);
        const uint32_t in4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i0 = (hh * MYC + c) * 8 + 2 * e;
          const float2 t = __ffma2_rn(make_float2(bf16_lo(in4[e]), bf16_hi(in4[e])), rs2, nm2);
          const float2 y = __ffma2_rn(t, gamma2[i0 / 2], beta2[i0 / 2]);
          mine[c * 4 + e] = tc::pack_bf16x2(y.x, y.y);
        }
      }
      // The other thread of this row has read both halves once it reaches the
      // pair barrier; then each thread writes its own half back.
      pair_sync(q4);
#pragma unroll
      for (int c = 0; c < MYC; ++c)
        *(uint4*)chunk_at(hh * MYC + c) =
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
        for (int t = 0; t < HPT; ++t) {
          const int head = hh * HPT + t;
          if (head < H)
            p.bias32[(bb * H + head) * NN + rc] = keep ? bsum[t] * kLog2e : -INFINITY;
        }
      }
    }
  } else if (warp < 2 * kWorkers / 32) {
    // ---------------- epilogue: cell row r = TMEM lane, column half hh
    const int ew = warp - kWorkers / 32;
    const int q4 = ew & 3, hh = ew >> 2;
    // Epilogue: each 32-row x 32-column chunk goes TMEM -> registers -> bf16 in a
    // swizzled smem staging tile -> one TMA store (full 64-byte row segments;
    // rows past the last cell are clipped by the tensor bounds). The two warps
    // of a lane quarter split every section (q, k, v, g) in column halves when
    // a section has two or more 32-column chunks (both then carry the same
    // sigmoid load), else take one section each; accumulator half nh (q|k or
    // v|g) is released as soon as both warps have read it.
    uint8_t* stg0 = smem + S::OFF_STG + ew * 2 * STG_BYTES;
    int nst = 0;                                  // TMA stores issued by this warp
    constexpr int CPS = S::CPS;
    constexpr int HALFC = CPS >= 2 ? CPS / 2 : 1;   // chunks per section per warp
    // Section and column (within the section) of this warp's chunk cw of
    // accumulator half nh.
    auto chunk_sect = [&](int nh, int cw) { return CPS >= 2 ? nh * 2 + cw / HALFC : nh * 2 + hh; };
    auto chunk_col = [&](int cw) { return CPS >= 2 ? (hh * HALFC + cw % HALFC) * 32 : 0; };
    auto epilogue = [&](int it) -> bool {
      const int tile = p.tile0 + blockIdx.x + it * gridDim.x;
      const int row0 = tile * BM + q4 * 32;
#pragma unroll 1
      for (int nh = 0; nh < 2; ++nh) {
        if (!warp_wait_or_abort(&bars->acc_full[nh], it & 1, ab)) return false;
        tc::tc_fence_after();
        // Half-chunk k (16 columns) of the 2 CPS this warp drains from
        // accumulator half nh. The load of half-chunk k + 1 is in flight while
        // half-chunk k is converted.
        auto hc_addr = [&](int k) {
          const int cw = k >> 1;
          return tc::tmem_addr(tmem, q4 * 32, chunk_sect(nh, cw) * D + chunk_col(cw) + (k & 1) * 16);
        };
        uint32_t accb[2][16];
        tc::tmem_ld16(hc_addr(0), accb[0]);
#pragma unroll
        for (int k = 0; k < 2 * CPS; ++k) {
          const int cw = k >> 1;
          const int sect = chunk_sect(nh, cw);
          const int col0 = chunk_col(cw);                    // within the section
          tc::tmem_ld_wait();
          if (k + 1 < 2 * CPS) tc::tmem_ld16(hc_addr(k + 1), accb[(k + 1) & 1]);
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
          } else if (sect == 2) {
            // v in fp16 (the resident Wv rows carry the power of 2 that keeps
            // |v| below 2^15 for any input).
#pragma unroll
            for (int e = 0; e < 8; ++e)
              packed[e] = cvt_f16x2(__uint_as_float(acc[2 * e]), __uint_as_float(acc[2 * e + 1]));
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
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, S::TMEM_COLS);
}

template <int D, int H>
cudaError_t launch(int grid, cudaStream_t s, bool pdl, const Maps& m, const Params& p,
                   const Consts& c) {
  return launch_pdl(pdl, ln_proj_tc<D, H>, dim3(grid), dim3(kThreads), Shape<D>::SMEM, s, m.x, m.w, m.q,
                    m.k, m.v, m.g, p, c);
}

template <int D, int H>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(ln_proj_tc<D, H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Shape<D>::SMEM);
}

}  // namespace k1

#define TRI_K1_SHAPES(X) X(32, 1) X(32, 2) X(64, 1) X(64, 2) X(64, 4) X(128, 2) X(128, 4) X(128, 8)

cudaError_t k1_init() {
  cudaError_t e = cudaSuccess;
#define X(D, H) if (e == cudaSuccess) e = k1::set_smem<D, H>();
  TRI_K1_SHAPES(X)
#undef X
  return e;
}

cudaError_t k1_launch(int D, int h, int grid, cudaStream_t s, bool pdl, const k1::Maps& m,
                      const k1::Params& p, const k1::Consts& c) {
#define X(DD, HH) if (D == DD && h == HH) return k1::launch<DD, HH>(grid, s, pdl, m, p, c);
  TRI_K1_SHAPES(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace tri_tc
