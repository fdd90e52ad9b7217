// Compile-time shapes of the bf16 tensor-core kernels: tile sizes, shared
// memory layout, tensor-memory columns and thread counts for each supported
// pair dimension D (32, 64, 128) and head dimension d (16, 32, 64).
//
// Plain C++ (no CUDA types), so that host code and the resource checks can
// read the same numbers the kernels are built with.
#pragma once

#include <stdint.h>

namespace tri_tc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxD = 128;     // largest pair dimension
constexpr int kMaxH = 8;       // most heads (D = 128, d = 16)

constexpr bool tc_shape_ok(int D, int h) {
  return (D == 32 || D == 64 || D == 128) && h >= 1 && D % h == 0 &&
         (D / h == 16 || D / h == 32 || D / h == 64);
}

constexpr uint32_t align_up(uint32_t a, uint32_t b) { return (a + b - 1) / b * b; }

// A channel row of D bf16 values is staged as K-halves of up to 64 channels;
// each half's rows are swizzled over their own length (32, 64 or 128 bytes, the
// TMA swizzle of the same name).
template <int D>
struct Channels {
  static constexpr int XSW = D >= 64 ? 128 : 2 * D;   // bytes per row of one half
  static constexpr int HC = XSW / 2;                  // channels per half
  static constexpr int KH = D / HC;                   // halves (1 or 2)
  static constexpr int CH16 = XSW / 16;               // 16-byte chunks per half row
  static constexpr int KSTEPS_PER_HALF = XSW / 32;    // 16-channel MMA K steps per half
};

// K1: LayerNorm + the q|k|v|g projection, 128-cell tiles.
namespace k1 {
constexpr int BM = 128;
constexpr int kWorkers = 256;                         // LayerNorm and epilogue threads
constexpr int kThreads = 2 * kWorkers + 64;
constexpr int kTmaWarp = 16, kMmaWarp = 17;
constexpr uint32_t STG_BYTES = 32 * 64;               // one 32 x 32 bf16 staging tile
template <int D>
struct Shape : Channels<D> {
  using C = Channels<D>;
  static constexpr int NQ = 4 * D;                    // q|k|v|g accumulator columns
  static constexpr int NHALF = 2 * D;                 // one accumulator half: q|k or v|g
  static constexpr int CPS = D / 32;                  // 32-column chunks per section
  static constexpr uint32_t X_HALF = BM * C::XSW;
  static constexpr uint32_t X_BYTES = C::KH * X_HALF;
  static constexpr uint32_t W_HALF = NQ * C::XSW;
  static constexpr uint32_t W_BYTES = C::KH * W_HALF;
  static constexpr uint32_t OFF_W = 0;
  static constexpr uint32_t OFF_X = align_up(W_BYTES, 1024);
  static constexpr uint32_t OFF_STG = OFF_X + 2 * X_BYTES;   // per epilogue warp: 2 tiles
  static constexpr uint32_t OFF_BAR = OFF_STG + 8 * 2 * STG_BYTES;
  static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;     // + alignment slack
  static constexpr int TMEM_COLS = NQ < 32 ? 32 : NQ;
};
}  // namespace k1

// K2: line attention. A work unit is (b, head, R lines, 128 queries); keys
// stream in 64-key sub-tiles.
namespace k2 {
constexpr int BQ = 128;                 // queries per unit
constexpr int BK = 64;                  // keys per sub-tile (one S buffer)
constexpr int B_STAGES = 3;             // bias sub-tile ring
constexpr int KV_STAGES_MAX = 4;        // K/V stage ring (barrier slots)
constexpr int TM_S1 = 64, TM_O = 128;   // per line: S0 | S1 | O
constexpr uint32_t BIAS_BYTES = BQ * BK * 2;
template <int DH>
struct Shape {
  // d = 64 fits two lines in tensor memory (S0 | S1 | O = 192 columns each).
  static constexpr int R = DH == 64 ? 2 : 3;
  // Keys per K/V stage: one sub-tile. A stage is released as soon as the P V
  // of its sub-tile completes, so four stages keep the copies three to four
  // sub-tiles ahead of the MMAs (two for d = 64, where shared memory is short).
  static constexpr int KVK = 64;
  static constexpr int KV_STAGES = DH == 64 ? 2 : 4;
  static constexpr int SPS = KVK / BK;                // sub-tiles per stage
  static constexpr int SW = 2 * DH;                   // row bytes = swizzle span of Q/K/V/O tiles
  static constexpr int kIssuers = R;
  static constexpr int kSoftmaxWarps = 4 * R;
  static constexpr int kThreads = 128 + 128 * R;
  // Registers: the control warpgroup lowers to kRegsCtl and the softmax
  // warpgroups raise to kRegsSoftmax; 32 (4 kRegsCtl + 4 R kRegsSoftmax) must
  // not exceed the registers the block is launched with.
  static constexpr int kRegsCtl = 48;
  static constexpr int kRegsSoftmax = R == 3 ? 152 : 216;
  static constexpr int kTmemPerRow = TM_O + (DH > 32 ? DH : 32);
  static constexpr uint32_t Q_BYTES = BQ * DH * 2;
  static constexpr uint32_t KVT_BYTES = KVK * DH * 2;   // K or V of one line, one stage
  static constexpr uint32_t KV_STAGE = R * 2 * KVT_BYTES;
  static constexpr uint32_t HALF_KV = BK * DH * 2;      // one sub-tile inside a K/V tile
  static constexpr uint32_t OST_BYTES = 32 * DH * 2;    // o staging per softmax warp
  static constexpr uint32_t OFF_Q = 0;                  // [2][R] Q tiles
  static constexpr uint32_t OFF_KV = OFF_Q + 2 * R * Q_BYTES;
  static constexpr uint32_t OFF_BIAS = OFF_KV + KV_STAGES * KV_STAGE;
  static constexpr uint32_t OFF_OST = OFF_BIAS + B_STAGES * BIAS_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_OST + kSoftmaxWarps * OST_BYTES;
  static constexpr uint32_t SMEM = OFF_BAR + 512 + 1024;
  static_assert(OFF_KV % 1024 == 0 && OFF_BIAS % 1024 == 0 && OFF_OST % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(R * kTmemPerRow <= 512, "tensor memory holds R lines");
  static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};
}  // namespace k2

// K3: gate product + output projection, 128-cell tiles.
namespace k3 {
constexpr int BM = 128;
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr uint32_t STG_BYTES = 32 * 64;
template <int D>
struct Shape : Channels<D> {
  using C = Channels<D>;
  static constexpr uint32_t T_HALF = BM * C::XSW;
  static constexpr uint32_t T_BYTES = C::KH * T_HALF;     // a g or o tile
  static constexpr uint32_t W_HALF = D * C::XSW;
  static constexpr uint32_t W_BYTES = C::KH * W_HALF;     // Wo
  static constexpr uint32_t OFF_W = 0;
  static constexpr uint32_t OFF_G = align_up(W_BYTES, 1024);   // g tiles [2]; become the A operand
  static constexpr uint32_t OFF_O = OFF_G + 2 * T_BYTES;       // o tiles [2]
  static constexpr uint32_t OFF_STG = OFF_O + 2 * T_BYTES;     // [4 warps][2]
  static constexpr uint32_t OFF_BO = OFF_STG + 4 * 2 * STG_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_BO + D * 4;
  static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
  static constexpr int TMEM_COLS = 2 * D < 32 ? 32 : 2 * D;    // two accumulators
};
}  // namespace k3

}  // namespace tri_tc
