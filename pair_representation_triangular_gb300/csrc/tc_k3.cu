// K3 of the bf16 tensor-core path: g * o formed in shared memory as the A
// operand of the output projection GEMM (M = 128 cells, N = K = D); the
// epilogue adds bo and stores bf16. Tiles are 128 cells in memory order, or 128
// rows of one grid column (the host-buffer forward of the ending node).
//
// Passages followed: POPCORNBENCH "Kimi-K2.6 l2_p6", forward op list steps
// 17-18 (gate product, output projection) and the layer definitions (the
// output projection carries a bias).
#include "tc_device.cuh"
#include "tc_kernels.cuh"

namespace tri_tc {
namespace k3 {

struct Bars {
  uint64_t w_full, in_full[2], in_empty[2], a_ready[2], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort;
};

// TMA coordinates (x, y, z) of tile `tile` after the channel coordinate.
struct TileAt { int x, y, z; };
__device__ __forceinline__ TileAt tile_at(const Params& p, int tile) {
  if (!p.cols) return {tile * BM, 0, 0};
  const int line = tile / p.tpl;
  return {(tile - line * p.tpl) * BM, line % p.N, line / p.N};
}

// Persistent: CTA c serves tiles c, c + G, ...; Wo (D x D bf16) stays in
// shared memory. Warps 0-3 form g * o (one cell row per thread), warps 4-7
// drain the accumulator (TMEM lane quarter = warp % 4), warp 8 TMA, warp 9 MMA:
// the gate product of tile t + 1 is formed while the epilogue drains tile t.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
gate_out_tc(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_o,
            const __grid_constant__ CUtensorMap map_wo, const __grid_constant__ CUtensorMap map_out,
            const Params p) {
  using S = Shape<D>;
  constexpr int XSW = S::XSW, CH16 = S::CH16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = (Bars*)(smem + S::OFF_BAR);
  float* s_bo = (float*)(smem + S::OFF_BO);
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
  for (int i = tid; i < D; i += kThreads) s_bo[i] = p.bo[i];
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
  int issued = 0;
  pdl_trigger();
  // g, o and out belong to earlier kernels on the stream; only Wo and bo are
  // read before the previous kernel's completion.
  if (warp != kTmaWarp) pdl_wait();

  if (warp == kTmaWarp) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&map_g);
      tc::tma_prefetch_desc(&map_o);
      tc::tma_prefetch_desc(&map_wo);
      tc::mbar_arrive_expect_tx(&bars->w_full, S::W_BYTES);
      for (int kh = 0; kh < S::KH; ++kh)
        tc::tma_load_2d(smem + S::OFF_W + kh * S::W_HALF, &map_wo, &bars->w_full, kh * S::HC, 0);
      pdl_wait();
      for (int it = 0; it < my_tiles; ++it) {
        const int b = it & 1;
        if (it >= 2 && !wait_or_abort(&bars->in_empty[b], ((it >> 1) - 1) & 1, ab)) break;
        const TileAt at = tile_at(p, p.tile0 + blockIdx.x + it * gridDim.x);
        uint8_t* gs = smem + S::OFF_G + b * S::T_BYTES;
        uint8_t* os = smem + S::OFF_O + b * S::T_BYTES;
        tc::mbar_arrive_expect_tx(&bars->in_full[b], 2 * S::T_BYTES);
        for (int kh = 0; kh < S::KH; ++kh) {
          tc::tma_load_4d(gs + kh * S::T_HALF, &map_g, &bars->in_full[b], kh * S::HC, at.x, at.y, at.z);
          tc::tma_load_4d(os + kh * S::T_HALF, &map_o, &bars->in_full[b], kh * S::HC, at.x, at.y, at.z);
        }
        issued = it + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, D, 0, 0);
      constexpr uint32_t swm = swz_mode(XSW);
      const uint32_t w0 = tc::smem_addr(smem + S::OFF_W);
      bool ok = wait_or_abort(&bars->w_full, 0, ab);
      for (int it = 0; ok && it < my_tiles; ++it) {
        const int b = it & 1;
        if (!wait_or_abort(&bars->a_ready[b], (it >> 1) & 1, ab)) break;
        if (it >= 2 && !wait_or_abort(&bars->acc_empty[b], ((it >> 1) - 1) & 1, ab)) break;
        tc::tc_fence_after();
        const uint32_t a0 = tc::smem_addr(smem + S::OFF_G + b * S::T_BYTES);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kh = ks / S::KSTEPS_PER_HALF, kin = ks % S::KSTEPS_PER_HALF;
          tc::mma_ss(tmem + b * D,
                          tc::smem_desc(a0 + kh * S::T_HALF + kin * 32, 16, 8 * XSW, swm),
                          tc::smem_desc(w0 + kh * S::W_HALF + kin * 32, 16, 8 * XSW, swm), idesc,
                          ks > 0);
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
      uint8_t* gs = smem + S::OFF_G + b * S::T_BYTES;
      const uint8_t* os = smem + S::OFF_O + b * S::T_BYTES;
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        const uint32_t off = (c / CH16) * S::T_HALF + swz(r, c % CH16, XSW);
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
    uint8_t* const stg0 = smem + S::OFF_STG + q4 * 2 * STG_BYTES;
    int nst = 0;                                  // TMA stores issued by this warp
    constexpr int NCH = D / 32;
    for (int it = 0; it < my_tiles; ++it) {
      const int b = it & 1;
      if (!warp_wait_or_abort(&bars->acc_full[b], (it >> 1) & 1, ab)) break;
      tc::tc_fence_after();
      const TileAt at = tile_at(p, p.tile0 + blockIdx.x + it * gridDim.x);
      // Chunk ch + 1 is loaded from TMEM while chunk ch is converted and stored.
      uint32_t accb[2][32];
      tc::tmem_ld32(tc::tmem_addr(tmem, q4 * 32, b * D), accb[0]);
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        tc::tmem_ld_wait();
        if (ch + 1 < NCH)
          tc::tmem_ld32(tc::tmem_addr(tmem, q4 * 32, b * D + (ch + 1) * 32), accb[(ch + 1) & 1]);
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
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, S::TMEM_COLS);
}

template <int D>
cudaError_t launch(int grid, cudaStream_t s, bool pdl, const Maps& m, const Params& p) {
  return launch_pdl(pdl, gate_out_tc<D>, dim3(grid), dim3(kThreads), Shape<D>::SMEM, s, m.g, m.o, m.wo,
                    m.out, p);
}

template <int D>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(gate_out_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Shape<D>::SMEM);
}

}  // namespace k3

cudaError_t k3_init() {
  cudaError_t e = k3::set_smem<32>();
  if (e == cudaSuccess) e = k3::set_smem<64>();
  if (e == cudaSuccess) e = k3::set_smem<128>();
  return e;
}

cudaError_t k3_launch(int D, int grid, cudaStream_t s, bool pdl, const k3::Maps& m,
                      const k3::Params& p) {
  switch (D) {
    case 32: return k3::launch<32>(grid, s, pdl, m, p);
    case 64: return k3::launch<64>(grid, s, pdl, m, p);
    case 128: return k3::launch<128>(grid, s, pdl, m, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tri_tc
