// K2 of the bf16 tensor-core path: flash-style line attention with the pair
// bias, the mask and the softmax, plus its small companions:
//
//   row_attn_tc  persistent: a work unit is (b, head t, R lines, 128 queries)
//                streaming 64-key tiles. Lines are grid rows (starting node)
//                or columns (ending node); only the tensor maps tell them
//                apart. S = Q K^T goes to TMEM; one softmax warpgroup per line
//                adds the shared fp16 bias tile, drops masked keys and writes
//                P = 2^x in fp16 over S; O += P V (fp16 operands, fp32
//                accumulator) accumulates in TMEM. The
//                (B, N, h, N, N) logits never exist. Instantiated for d = 16,
//                32 and 64.
//   bias_rows    the attention's fp16 bias plane (B, h, N, Nb), indexed
//                [query, key] along the attended line: each (head, query) row
//                minus its largest entry (the softmax is unchanged, and fp16
//                is then precise where the weights are large).
//   mask_summary / mask_summary_cols
//                keep bits and a "keeps some key" flag of every line.
//
// Passages followed: POPCORNBENCH "Kimi-K2.6 l2_p6", forward op list steps
// 10-16 (scaled logits, pair bias, mask, softmax, weighted sum of v);
// "FW-GLM-5-1 l2_p6", quoted Model.forward (the mask broadcast).
#include "tc_device.cuh"
#include "tc_kernels.cuh"

namespace tri_tc {
namespace k2 {

template <int R>
struct Bars {
  uint64_t q_full[2], q_empty[2], kv_full[KV_STAGES_MAX], kv_empty[KV_STAGES_MAX];
  uint64_t b_full[B_STAGES], b_empty[B_STAGES];
  // s_ready and p_full follow the S/P buffer (sub-tile parity): a warp with no
  // live lanes runs ahead, and its arrivals for sub-tile c + 1 must not complete
  // the phase of sub-tile c.
  uint64_t s_ready[R][2], p_full[R][2], p_free[R][2], o_free[R], drain[R];
  uint32_t tmem_base;
  int abort;
  // Key sub-tiles of unit ui in slot ui & 7, written by the producer before the
  // unit's first copies (the consumers read it after waiting on one of them:
  // the MMA warps on the unit's Q, the softmax on its first bias sub-tile).
  // The producer rewrites a slot only after the MMAs of the unit six places
  // on have been issued, which needs the softmax four units on, so every
  // reader of the slot is done with it.
  int unit_kt[8];
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

// Key sub-tiles of a unit: the row-key reading skips the trailing sub-tiles
// that every line of the unit drops (a line that keeps no key needs all of
// them); the query-key reading takes all KT.
template <int R>
__device__ __forceinline__ int unit_tiles(const Unit& u, const Params& p, int KT) {
  if (p.mask_mode == TRI_ATTN_MASK_QUERY_KEY) return KT;
  int t = 1;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int a = u.rg * R + r;
    if (a < p.N) t = max(t, __ldg(p.line_tiles + (long long)u.b * p.N + a));
  }
  return t;
}

// Position in a stream of sub-tiles: global sub-tile c, its unit ui and key
// sub-tile kt, the K/V stage slot and phase, and the bias slot and phase,
// advanced without dividing. KTu: the sub-tiles of unit ui.
struct SubIt {
  int c, ui, kt, kvs, kvph, bs, bph;
};
template <int SPS, int KV_STAGES>
__device__ __forceinline__ void advance(SubIt& it, int KTu) {
  ++it.c;
  const bool stage_end = (it.kt % SPS) == SPS - 1 || it.kt == KTu - 1;
  if (++it.kt == KTu) { it.kt = 0; ++it.ui; }
  if (stage_end && ++it.kvs == KV_STAGES) { it.kvs = 0; it.kvph ^= 1; }
  if (++it.bs == B_STAGES) { it.bs = 0; it.bph ^= 1; }
}

// The softmax's position in its sub-tile stream: global sub-tile c and the
// bias slot and phase.
struct SoftIt {
  int c, bs, bph;
};
__device__ __forceinline__ void advance_soft(SoftIt& it) {
  ++it.c;
  if (++it.bs == B_STAGES) { it.bs = 0; it.bph ^= 1; }
}

// Real-key bits of word w (keys 32w..32w+31 of a sub-tile with `left` keys left).
__device__ __forceinline__ uint32_t real_bits(int left, int w) {
  const int n = left - 32 * w;
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// The 64 fp16 biases of a sub-tile row (brow: the row's swizzled base, 16-byte
// chunk q, keys 8q .. 8q + 7, at brow ^ (q << 4)).
__device__ __forceinline__ void load_bias(uint32_t brow, uint4 (&bh)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) bh[q] = tc::lds128(brow ^ (q << 4));
}

// One 64-key sub-tile row, every lane live: P = 2^(S + bias) with S (fp32
// bits, sv) in log2 units (the reference of the exponentials is 0). Each key
// pair of S is rounded to an fp16 pair, the fp16 bias pair added and 2^x taken
// of both halves at once; P leaves as 32 fp16 pairs (the A operand of the P V
// MMA) and the return value is their sum as one fp16 pair: four running sums,
// each taking every fourth pair as it is produced, then added pairwise.
__device__ __forceinline__ uint32_t p_tile_fast(const uint32_t (&sv)[2 * BK / 2], const uint4 (&bh)[8],
                                                uint32_t (&pk)[BK / 2]) {
  uint32_t acc[4];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t hw[4] = {bh[q].x, bh[q].y, bh[q].z, bh[q].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = q * 4 + e;
      pk[m] = ex2_f16x2(hadd2(cvt_f16x2(__uint_as_float(sv[2 * m]), __uint_as_float(sv[2 * m + 1])), hw[e]));
      acc[e] = q == 0 ? pk[m] : hadd2(acc[e], pk[m]);
    }
  }
  return hadd2(hadd2(acc[0], acc[1]), hadd2(acc[2], acc[3]));
}

// P of a 64-key sub-tile row of a lane that is not live: 1 on every real key
// of a uniform row or query (w0, w1: the sub-tile's real-key bits), else 0
// (fp16 pairs).
__device__ __forceinline__ void p_tile_const(uint32_t w0, uint32_t w1, uint32_t (&pk)[BK / 2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t w = h ? w1 : w0;
    if (w == 0u || w == 0xffffffffu) {
      const uint32_t v = w ? 0x3C003C00u : 0u;
#pragma unroll
      for (int k = 0; k < 16; ++k) pk[16 * h + k] = v;
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        pk[16 * h + k] = (((w >> (2 * k)) & 1u) ? 0x3C00u : 0u) |
                         (((w >> (2 * k + 1)) & 1u) ? 0x3C000000u : 0u);
    }
  }
}

// A query row whose sum l left [2^-6, 2^100] is recomputed exactly on the
// CUDA cores: a logit reached 2^16 in P = 2^x (fp16 holds P below 65504, and
// an infinite or undefined P makes l infinite or NaN), or every key it keeps
// lies more than 6 below 0 in log2 units, where fp16 P loses relative
// precision (subnormal below 2^-14) and the fp16 bias plane's rounding is no
// longer small: the row's largest bias may sit at a key the line drops (the
// row-key reading). Two passes over the line's keys, the first for the row max m, the
// second for l = sum 2^(x - m) and o = sum 2^(x - m) v / l, in fp32 with the
// fp32 bias. qrow: the row's q (head t); kl, vl: key 0 of the line's k and v
// (head t), sx: the stride between keys; brow: the bias of the row's key 0 in
// the fp32 cell-order plane and bs the stride between keys; keys come from the
// line's mask bits (row reading; mrow) or from the finite biases (query
// reading, mrow = null: the plane holds -inf for dropped keys); v is fp16
// times 1 / v_unscale. o leaves as d / 2 bf16 pairs in the lane's row of the
// swizzled staging tile at stg (rows of 2 d bytes).
template <int DH>
__device__ __noinline__ void exact_row(const __nv_bfloat16* qrow, const __nv_bfloat16* kl,
                                       const __half* vl, float v_unscale, long long sx,
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
    const __half* vr = vl + (long long)kk * sx;
#pragma unroll
    for (int e = 0; e < DH; ++e) o[e] = fmaf(w, __half2float(vr[e]), o[e]);
  }
  const float inv = l > 0.f ? v_unscale / l : 0.f;
#pragma unroll
  for (int qc = 0; qc < DH / 8; ++qc) {
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w4[e] = tc::pack_bf16x2(o[8 * qc + 2 * e] * inv, o[8 * qc + 2 * e + 1] * inv);
    *(uint4*)(stg + swz(lane, qc, 2 * DH)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
}

// Persistent: CTA c serves work units unit0 + c, + G, ... A unit is (b, head
// t, R lines, 128 queries), R = 3 (d = 16, 32) or 2 (d = 64, whose three
// lines would not fit tensor memory); it streams 64-key sub-tiles, all of
// them or, under the row-key reading, up to the last one that some line of the
// unit keeps a key of. The K and V tiles of the R lines arrive one sub-tile per
// stage, in a ring of four stages (two for d = 64, where shared memory is
// short); the fp16 bias sub-tile they share has a ring of its own. Warpgroup 0: warp 0 TMA, warp
// 1 + r issues the MMAs of line r (both roles run as whole warps; one elected
// lane issues); warpgroup 1 + r runs the softmax of line r, with registers
// moved to it from warpgroup 0 (setmaxnreg). Tensor memory per line: S0 | S1
// (64 fp32 columns each) | O (d columns from column 128).
// Softmax warpgroup r owns line r; sub-tile c's S = Q K^T lands in the line's
// S buffer c & 1 in log2 units (q carries the factor log2(e)/sqrt(d)), and the
// softmax rounds S to fp16 pairs, adds the fp16 bias pair, drops masked keys
// and writes P = 2^x (fp16, two per 32-bit column) over it in one pass, with
// one packed 2^x per key pair; the line's MMA warp then issues O += P V(c)
// (V in fp16) and S(c + 2) into the same buffer. The reference of the
// exponentials is fixed at 0: no max is taken; fp16 P holds 2^x with 11-bit
// precision for -14 <= x < 16, beyond the logits of layer-normalised
// activations (the bias rows are stored minus their maximum); a query row
// whose sum l ends outside [2^-6, 2^100] is recomputed exactly in the unit
// epilogue (exact_row). A unit's o = O / l is read and stored after the
// next unit's first sub-tile, which hides the completion of the unit's last
// P V.
template <int DH>
__global__ void __launch_bounds__(Shape<DH>::kThreads, 1)
row_attn_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_b,
            const __grid_constant__ CUtensorMap map_o, const Params p) {
  using S = Shape<DH>;
  constexpr int R = S::R, SPS = S::SPS, SW = S::SW, KV_STAGES = S::KV_STAGES;
  constexpr int kIssuers = S::kIssuers, kSoftmaxWarps = S::kSoftmaxWarps;
  constexpr int kRegsCtl = S::kRegsCtl, kRegsSoftmax = S::kRegsSoftmax;
  constexpr int kTmemPerRow = S::kTmemPerRow;
  constexpr uint32_t Q_BYTES = S::Q_BYTES, KVT_BYTES = S::KVT_BYTES, KV_STAGE = S::KV_STAGE;
  constexpr uint32_t HALF_KV = S::HALF_KV, OST_BYTES = S::OST_BYTES;
  constexpr uint32_t OFF_Q = S::OFF_Q, OFF_KV = S::OFF_KV, OFF_BIAS = S::OFF_BIAS;
  constexpr uint32_t OFF_OST = S::OFF_OST, OFF_BAR = S::OFF_BAR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars<R>* bars = (Bars<R>*)(smem + OFF_BAR);
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
      tc::mbar_init(&bars->b_empty[s], 32 * kSoftmaxWarps);   // every softmax thread arrives
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
  // Every input of the attention comes from the kernels before it on the
  // stream, and o may still be read by the previous forward's output kernel.
  pdl_trigger();
  pdl_wait();

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
        const int KTu = unit_tiles<R>(un, p, KT);
        if (ui >= 2 && !warp_wait_or_abort(&bars->q_empty[qb], ((ui >> 1) - 1) & 1, ab)) break;
        if (elect_one()) {
          bars->unit_kt[ui & 7] = KTu;
          tc::mbar_arrive_expect_tx(&bars->q_full[qb], R * Q_BYTES);
          for (int r = 0; r < R; ++r)
            tc::tma_load_4d(smem + OFF_Q + (qb * R + r) * Q_BYTES, &map_q, &bars->q_full[qb],
                            un.t * DH, un.j0, a0 + r, un.b);
        }
        __syncwarp();
        q_issued = ui + 1;
        for (int kt = 0; kt < KTu; ++kt) {
          if (kt % SPS == 0) {
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
    } else if (warp - 1 < R) {
      // ---------------- MMA issuer of line r = warp - 1 (whole warp; one elected lane
      // issues). With R = 2, warp 3 has no role and goes straight to the teardown.
      // The line index and the tensor-memory base are broadcast from lane 0 so
      // that the compiler sees every MMA operand as warp-uniform (uniform
      // registers: the elected lane issues without a per-lane loop).
      const int r = __shfl_sync(0xffffffffu, warp - 1, 0);
      const uint32_t tr = __shfl_sync(0xffffffffu, tmem, 0) + r * kTmemPerRow;
      constexpr uint32_t id_qk = tc::idesc_bf16_f32(128, BK, 0, 0);
      // P (fp16, tensor memory) times V (fp16): both operands fp16.
      constexpr uint32_t id_pv = tc::idesc_f16_f32(128, DH, 0, 1);
      // Descriptors of this line's first Q tile and first K tile; every other
      // operand sits a multiple of 16 bytes further (the start-address field
      // holds address / 16 and stays below 2^14).
      const uint64_t dq0 = tc::smem_desc(tc::smem_addr(smem + OFF_Q + r * Q_BYTES), 16, 8 * SW, swz_mode(SW));
      const uint64_t dk0 =
          tc::smem_desc(tc::smem_addr(smem + OFF_KV + r * 2 * KVT_BYTES), 16, 8 * SW, swz_mode(SW));
      // The sub-tiles of a cursor's unit, published by the producer before the
      // unit's Q copy, which the S cursor (never behind the P V one) has waited on.
      auto unit_kt = [&](const SubIt& it) -> int { return *(volatile int*)&bars->unit_kt[it.ui & 7]; };
      auto qk = [&](const SubIt& it) -> bool {
        const int c = it.c;
        if (it.kt == 0 && !warp_wait_or_abort(&bars->q_full[it.ui & 1], (it.ui >> 1) & 1, ab)) return false;
        if (it.kt % SPS == 0 && !warp_wait_or_abort(&bars->kv_full[it.kvs], it.kvph, ab)) return false;
        tc::tc_fence_after();
        if (elect_one()) {
          const uint64_t qd = dq0 + (uint64_t)(((it.ui & 1) * R * Q_BYTES) >> 4);
          const uint64_t kd = dk0 + (uint64_t)((it.kvs * KV_STAGE + (it.kt % SPS) * HALF_KV) >> 4);
#pragma unroll
          for (int ks = 0; ks < DH / 16; ++ks)
            tc::mma_ss(tr + (c & 1) * TM_S1, qd + 2 * ks, kd + 2 * ks, id_qk, ks > 0);
          tc::mma_commit(&bars->s_ready[r][c & 1]);
          if (it.kt == unit_kt(it) - 1) tc::mma_commit(&bars->q_empty[it.ui & 1]);
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
              dk0 + (uint64_t)((it.kvs * KV_STAGE + KVT_BYTES + (it.kt % SPS) * HALF_KV) >> 4);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            tc::mma_ts(tr + TM_O, tr + (c & 1) * TM_S1 + ks * 8, vd + SW * ks, id_pv,
                            (it.kt > 0 || ks > 0) ? 1u : 0u);
          tc::mma_commit(&bars->p_free[r][c & 1]);
          if (it.kt % SPS == SPS - 1 || it.kt == unit_kt(it) - 1) tc::mma_commit(&bars->kv_empty[it.kvs]);
        }
        __syncwarp();
        return true;
      };
      bool ok = true;
      SubIt itq{0, 0, 0, 0, 0, 0, 0}, itp{0, 0, 0, 0, 0, 0, 0};
      for (; ok && itq.c < 2 && itq.ui < my_units; advance<SPS, KV_STAGES>(itq, unit_kt(itq))) ok = qk(itq);
      for (; ok && itp.ui < my_units; advance<SPS, KV_STAGES>(itp, unit_kt(itp))) {
        ok = pv(itp);
        if (ok && itq.ui < my_units) {
          ok = qk(itq);
          advance<SPS, KV_STAGES>(itq, unit_kt(itq));
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
    // give the keys this lane keeps, with its first two words. Loaded one unit
    // ahead.
    auto unit_loads = [&](const Unit& nu, unsigned& any, const uint32_t*& mrow, uint2& bits0) {
      const int nj = nu.j0 + jr, ni = nu.rg * R + r;
      const int mr = qk_mode ? nj : ni;
      // Queries past N produce nothing (their stores are clipped): they count
      // as keeping keys so that they never force the general path.
      any = mr < N ? tc::ldg_nc_u8_early(p.row_any + (long long)nu.b * N + mr) : (qk_mode ? 1u : 0u);
      mrow = p.mbits + ((long long)nu.b * N + (mr < N ? mr : 0)) * p.words;
      bits0 = tc::ldg_nc_v2_early(mrow);
    };
    unsigned nx_any = 0u;
    const uint32_t* nx_mrow = p.mbits;
    uint2 nx_bits0 = make_uint2(0u, 0u);
    // Units advance by digit-wise steps: cu is unit ui, pu the unit before it.
    Unit cu = decode_unit(p.unit0 + blockIdx.x, p), pu = cu;
    if (my_units > 0) unit_loads(cu, nx_any, nx_mrow, nx_bits0);
    // Unit epilogue: o = O / l once the unit's last P V has landed, staged in
    // shared memory and written by one TMA store per warp (queries past N are
    // clipped by the store; lines past N and warps whose 32 queries all lie
    // past N skip it).
    uint8_t* const ostg = smem + OFF_OST + sw * OST_BYTES;
    auto finish_unit = [&](const Unit& fu, int clast, float l) -> bool {
      if (!warp_wait_or_abort(&bars->p_free[r][clast & 1], (clast >> 1) & 1, ab)) return false;
      tc::tc_fence_after();
      uint32_t ov[DH];
      if constexpr (DH == 16) {
        tc::tmem_ld16(tb + TM_O, *(uint32_t(*)[16])ov);
      } else {
#pragma unroll
        for (int hc = 0; hc < DH / 32; ++hc)
          tc::tmem_ld32(tb + TM_O + 32 * hc, *(uint32_t(*)[32]) & ov[32 * hc]);
      }
      tc::tmem_ld_wait();
      // O is in registers: its columns may take the next unit's sums.
      tc::tc_fence_before();
      tc::mbar_arrive(&bars->o_free[r]);
      const int fi = fu.rg * R + r, fj = fu.j0 + (warp & 3) * 32;
      if (fi < N && fj < N) {
        // A query row has l in [2^-16, 2^100) unless its logits left that range
        // (a uniform row or query has l = its count of real keys): those rows
        // are recomputed exactly.
        const bool exact = fj + lane < N && !(l >= 0x1p-6f && l <= 0x1p100f);
        // l lies in [2^-6, 2^100]: the fast form is exact enough. V is stored
        // times a power of 2, taken out here.
        const float inv = __fdividef(p.v_unscale, l);
        uint32_t po[DH / 2];
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
          exact_row<DH>(p.q + base + (long long)a * p.sx, p.k + base, p.v + base, p.v_unscale, p.sx,
                    p.bias32 + plane + (p.ending ? (long long)a : (long long)a * N),
                    p.ending ? (long long)N : 1ll,
                    p.mask_mode == TRI_ATTN_MASK_QUERY_KEY
                        ? nullptr
                        : p.mbits + ((long long)fu.b * N + fi) * p.words,
                    N, ostg, lane);
        } else {
#pragma unroll
          for (int q = 0; q < DH / 8; ++q)
            *(uint4*)(ostg + swz(lane, q, SW)) =
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
    SoftIt its{0, 0, 0};                            // this warp's sub-tile stream
    float l_prev = 0.f;
    for (int ui = 0; ok && ui < my_units; ++ui) {
      const bool uni = nx_any == 0u;
      const uint32_t* mrow = nx_mrow;
      uint2 nbits = nx_bits0;
      Unit nu = cu;
      step_unit(nu, p);
      if (ui + 1 < my_units) unit_loads(nu, nx_any, nx_mrow, nx_bits0);
      float l_run = 0.f;
      // Warp-uniform unit state: whether any lane has a key-keeping query row.
      const bool unit_live = __any_sync(0xffffffffu, !uni);
      // The unit's key sub-tiles (KT until read after the first sub-tile's waits).
      int KTu = KT;
      for (int kt = 0; ok && kt < KTu; ++kt, advance_soft(its)) {
        const int c = its.c;
        const uint2 mb = nbits;
        if (kt + 1 < KTu) nbits = tc::ldg_nc_v2_early(mrow + 2 * (kt + 1));
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
        if (kt == 0) KTu = *(volatile int*)&bars->unit_kt[ui & 7];
        const bool any_live = unit_live && tile_keys;
        tc::tc_fence_after();
        const uint32_t tsb = tb + (c & 1) * TM_S1;     // S(c), then P(c) over it
        uint32_t tsum = 0u;                            // fp16 pair
        uint32_t pk[BK / 2];
        // The common sub-tile (every key real and kept) has a copy of its own
        // without the masking, which slowed it even when skipped.
        if (any_live && all_kept) {
          uint32_t sv[BK];
          uint4 bh[8];
          tc::tmem_ld64(tsb, sv);
          load_bias(brow, bh);
          tc::tmem_ld_wait();
          if (live)
            tsum = p_tile_fast(sv, bh, pk);
          else
            p_tile_const(uni ? rl0 : 0u, uni ? rl1 : 0u, pk);
        } else if (any_live) {
          uint32_t sv[BK];
          uint4 bh[8];
          tc::tmem_ld64(tsb, sv);
          load_bias(brow, bh);
          tc::tmem_ld_wait();
          // Dropped keys: S = -inf, which the bias add keeps at -inf (P = 0).
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            if (!((bw0 >> k) & 1u)) sv[k] = 0xff800000u;
            if (!((bw1 >> k) & 1u)) sv[32 + k] = 0xff800000u;
          }
          if (live)
            tsum = p_tile_fast(sv, bh, pk);
          else
            p_tile_const(uni ? rl0 : 0u, uni ? rl1 : 0u, pk);
        } else {
          // No lane of the warp keeps a key of this sub-tile: P is 1 on the real
          // keys of a uniform row or query, else 0.
          p_tile_const(uni ? rl0 : 0u, uni ? rl1 : 0u, pk);
        }
        tc::tmem_st32(tsb, pk);
        // The bias stage is read: release it (every softmax thread arrives).
        tc::mbar_arrive(&bars->b_empty[its.bs]);
        if (live) {
          l_run += f16x2_sum(tsum);
        } else if (uni) {
          l_run += (float)(__popc(rl0) + __popc(rl1));
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(&bars->p_full[r][c & 1]);
        if (kt == 0 && ui >= 1) {
          // The previous unit's epilogue, after this unit's first sub-tile.
          if (!finish_unit(pu, c - 1, l_prev)) { ok = false; break; }
        }
      }
      if (!ok) break;
      l_prev = l_run;
      pu = cu;
      cu = nu;
    }
    if (ok && my_units > 0) finish_unit(pu, its.c - 1, l_prev);
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
// block of C (32 contiguous bytes per key) through shared memory. Rows of up
// to 1024 keys are read once: every load of the row is issued before the
// maximum is taken (the ending node's 8-query block moves through shared
// memory whole). A row with every key dropped stays -inf.
constexpr int kBiasRowChunks = 8;           // keys read in one pass: 8 x 128
__global__ void __launch_bounds__(256)
bias_rows(const float* __restrict__ C, int N, int Nb, int ending, __half* __restrict__ P) {
  __shared__ float tile[8][kBiasRowChunks * 128 + 4];
  pdl_trigger();
  pdl_wait();
  const int a0 = blockIdx.x * 8;
  const long long plane = blockIdx.y;
  const float* Cp = C + plane * N * N;
  __half* Pp = P + plane * N * Nb;
  const int wq = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = a0 + wq;                          // this warp's row
  // Writes keys k .. k + 3 of the row (entries v minus the row maximum m).
  auto store4 = [&](int k, const float (&v)[4], float m) {
    __half hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) hv[e] = __float2half_rn(m == -INFINITY ? -INFINITY : v[e] - m);
    if (k + 3 < N) {                              // 8-byte store: Nb and k are multiples of 4
      *(uint2*)(Pp + (long long)a * Nb + k) = *(const uint2*)hv;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (k + e < N) Pp[(long long)a * Nb + k + e] = hv[e];
    }
  };
  if (N <= kBiasRowChunks * 128) {
    float v[kBiasRowChunks][4];
    if (ending) {
      // Thread i moves C[k][a0 + 4 (i & 1) .. + 3] for keys k = i / 2 + 128 c.
      const int qa = 4 * (threadIdx.x & 1);
#pragma unroll
      for (int c = 0; c < kBiasRowChunks; ++c) {
        const int kk = 128 * c + (threadIdx.x >> 1);
        if (128 * c < N) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            tile[qa + e][kk] = (kk < N && a0 + qa + e < N) ? Cp[(long long)kk * N + a0 + qa + e] : -INFINITY;
        }
      }
      __syncthreads();
#pragma unroll
      for (int c = 0; c < kBiasRowChunks; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          v[c][e] = 128 * c < N ? tile[wq][128 * c + 4 * lane + e] : -INFINITY;
    } else {
#pragma unroll
      for (int c = 0; c < kBiasRowChunks; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = 128 * c + 4 * lane + e;
          v[c][e] = (k < N && a < N) ? Cp[(long long)a * N + k] : -INFINITY;
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < kBiasRowChunks; ++c)
      m = fmaxf(fmaxf(m, fmaxf(v[c][0], v[c][1])), fmaxf(v[c][2], v[c][3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (a < N) {
#pragma unroll
      for (int c = 0; c < kBiasRowChunks; ++c)
        if (128 * c < N) store4(128 * c + 4 * lane, v[c], m);
    }
    return;
  }
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
        store4(k0 + 4 * lane, v, m);
      }
    }
    if (pass == 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
  }
}

// Leading 64-key sub-tiles a mask row needs: through its last kept key (last,
// -1 if none), or every sub-tile when it keeps none (its weights then spread
// over all real keys).
__device__ __forceinline__ int row_tiles(int last, int N) {
  return last < 0 ? (N + BK - 1) / BK : last / BK + 1;
}

// Mask rows (b, r): bit k of word k/32 is pair_mask[b, r, k] != 0 for k < N
// (0 beyond, up to `words` words), any[row] says whether the row keeps some key
// and tiles[row] how many leading sub-tiles it needs. A block takes 8 rows with
// 4 warps each (warp part p forms the words p, p + 4, ...); the parts' last
// kept keys are combined in shared memory.
constexpr int kMaskRowParts = 4;
__global__ void __launch_bounds__(256 * kMaskRowParts)
mask_summary(const int32_t* __restrict__ mask, int N, long long rows, int words,
             uint32_t* __restrict__ bits, unsigned char* __restrict__ any, int* __restrict__ tiles) {
  __shared__ int found[8][kMaskRowParts];
  pdl_trigger();
  pdl_wait();
  const int wp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rl = wp / kMaskRowParts, part = wp % kMaskRowParts;
  const long long row = (long long)blockIdx.x * 8 + rl;
  int last = -1;
  if (row < rows) {
    for (int wd = part; wd < words; wd += kMaskRowParts) {
      const int k = wd * 32 + lane;
      const bool keep = k < N && mask[row * N + k] != 0;
      const unsigned w = __ballot_sync(0xffffffffu, keep);
      if (w) last = wd * 32 + 31 - __clz(w);
      if (lane == 0) bits[row * words + wd] = w;
    }
  }
  if (lane == 0) found[rl][part] = last;
  __syncthreads();
  if (part == 0 && lane == 0 && row < rows) {
#pragma unroll
    for (int i = 1; i < kMaskRowParts; ++i) last = max(last, found[rl][i]);
    any[row] = last >= 0;
    tiles[row] = row_tiles(last, N);
  }
}

// Ending node: line (b, a) is column a of the mask (key k = grid row k). A
// block takes 32 columns of one batch, lane = column a; warp wp forms the
// words w = wp, wp + 32, ... (bit kk of word w: pair_mask[b, 32 w + kk, a] != 0,
// each of its 32 loads one coalesced 128-byte row segment across the warp),
// and the block combines the warps' last kept keys in shared memory. There are
// few blocks (one per 32 columns), so each has 32 warps.
constexpr int kMaskColWarps = 32;
__global__ void __launch_bounds__(32 * kMaskColWarps)
mask_summary_cols(const int32_t* __restrict__ mask, int N, int words, uint32_t* __restrict__ bits,
                  unsigned char* __restrict__ any, int* __restrict__ tiles) {
  __shared__ int found[kMaskColWarps][32];
  pdl_trigger();
  pdl_wait();
  const int cblocks = (N + 31) >> 5;
  const long long b = blockIdx.x / cblocks;
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  const int a = (int)(blockIdx.x % cblocks) * 32 + lane;
  int last = -1;                       // last kept key among this warp's words
  if (a < N) {
    const int32_t* col = mask + b * N * N + a;
    for (int w = wp; w < words; w += kMaskColWarps) {
      uint32_t word = 0;
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const int k = 32 * w + kk;
        if (k < N && col[(long long)k * N] != 0) word |= 1u << kk;
      }
      bits[(b * N + a) * words + w] = word;
      if (word) last = 32 * w + 31 - __clz(word);
    }
  }
  found[wp][lane] = last;
  __syncthreads();
  if (wp == 0 && a < N) {
#pragma unroll
    for (int i = 1; i < kMaskColWarps; ++i) last = max(last, found[i][lane]);
    any[b * N + a] = last >= 0;
    tiles[b * N + a] = row_tiles(last, N);
  }
}

template <int DH>
cudaError_t launch(int grid, cudaStream_t s, bool pdl, const Maps& m, const Params& p) {
  return launch_pdl(pdl, row_attn_tc<DH>, dim3(grid), dim3(Shape<DH>::kThreads), Shape<DH>::SMEM, s, m.q,
                    m.k, m.v, m.b, m.o, p);
}

template <int DH>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(row_attn_tc<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Shape<DH>::SMEM);
}

}  // namespace k2

cudaError_t k2_init() {
  cudaError_t e = k2::set_smem<16>();
  if (e == cudaSuccess) e = k2::set_smem<32>();
  if (e == cudaSuccess) e = k2::set_smem<64>();
  return e;
}

int k2_lines_per_unit(int d) {
  return d == 16 ? k2::Shape<16>::R : d == 32 ? k2::Shape<32>::R : k2::Shape<64>::R;
}

int k2_keys_per_stage(int d) {
  return d == 16 ? k2::Shape<16>::KVK : d == 32 ? k2::Shape<32>::KVK : k2::Shape<64>::KVK;
}

cudaError_t k2_launch(int d, int grid, cudaStream_t s, bool pdl, const k2::Maps& m,
                      const k2::Params& p) {
  switch (d) {
    case 16: return k2::launch<16>(grid, s, pdl, m, p);
    case 32: return k2::launch<32>(grid, s, pdl, m, p);
    case 64: return k2::launch<64>(grid, s, pdl, m, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t k2_mask_summary(const int32_t* mask, int B, int N, bool ending, int words,
                            uint32_t* bits, unsigned char* any, int* tiles, cudaStream_t s, bool pdl) {
  const long long rows = (long long)B * N;
  if (!ending)
    return launch_pdl(pdl, k2::mask_summary, dim3((unsigned)((rows + 7) / 8)), dim3(256 * k2::kMaskRowParts),
                      0, s, mask, N, rows, words, bits, any, tiles);
  const unsigned blocks = (unsigned)(B * (long long)((N + 31) / 32));
  return launch_pdl(pdl, k2::mask_summary_cols, dim3(blocks), dim3(32 * k2::kMaskColWarps), 0, s, mask, N,
                    words, bits, any, tiles);
}

cudaError_t k2_bias_rows(const float* C, int B, int h, int N, int Nb, bool ending, __half* P,
                         cudaStream_t s, bool pdl) {
  const dim3 grid((unsigned)((N + 7) / 8), (unsigned)(B * h));
  return launch_pdl(pdl, k2::bias_rows, grid, dim3(256), 0, s, C, N, Nb, ending ? 1 : 0, P);
}

}  // namespace tri_tc
