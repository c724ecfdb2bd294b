// gemm.cuh - host-side interface of the grouped GEMM kernels (gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

// Which contraction a launch performs; fixes the operand majorness and the
// epilogue.
enum class GemmKind : int {
  kFc1Act = 0,    // A = x_perm (K-major), B = W1 (N-major, 3-D); act epilogue
  kFc2 = 1,       // A = a (K-major),      B = W2 (N-major, 3-D); store
  kDgradAct = 2,  // A = dy_perm (K-major), B = W2^T (K-major, 3-D); dAct epilogue
  kDgrad = 3,     // A = dh (K-major),     B = W1^T (K-major, 3-D); store
  kWgrad = 4,     // A = act^T (M-major),  B = grad (N-major); ragged K
};

struct GemmArgs {
  const int32_t* offsets;  // [E+1] device
  int E;
  int M_cap;
  int K;                   // reduction length (ragged-row kinds)
  int N;                   // output columns
  int R;                   // output rows per expert (kWgrad)
  uint16_t* out;           // bf16 output
  long long ldo;           // output row stride, elements
  long long out_estride;   // elements between experts' outputs (kWgrad)
  uint16_t* out2;          // kFc1Act: H (optional)
  long long ldo2;
  const uint16_t* aux;     // kDgradAct: saved H
  long long ld_aux;
  int32_t* err;
  // kFc1Act with MXFP8 output (all NULL otherwise)
  uint8_t* mx_q;           // [M_cap, n] E4M3 codes of A (row-wise 1x32 blocks)
  uint8_t* mx_s;           // row-wise scales, MMA-tiled by 128-row tile start
  uint8_t* mx_qT;          // [n, M_cap] codes of A^T (32x1 blocks) or NULL
  uint8_t* mx_sT;          // [n, M_cap/32] scales of mx_qT
  int n_a;                 // columns of A (n)
  // kDgradAct, routed (probs != nullptr): the accumulator is dA' = dO W2^T
  // before the router probability p of the row's pair; the epilogue writes
  // dH = act'(H; p dA'), A' = p act(H) and the partial <dA', act(H)> of each
  // 128-column half tile
  const int32_t* pair_of_row;  // [M_cap] row -> pair (-1: pad row)
  const float* probs;          // [T*k] probability of each pair
  uint16_t* out3;              // A' [M_cap, ldo3] bf16
  long long ldo3;
  float* ds_part;              // [M_cap, ds_parts] fp32
  int ds_parts;
  // optional NVFP4 statistic, raised with atomicMax (the caller sets the
  // start value): kFc1Act max |A| of the bf16 A; kDgradAct max over 16-row
  // blocks (from each expert's first row) of |H16 dH| / 4 per dH column
  float* amax;
  // unit order inside an expert, set by launch_grouped_gemm: 0 = row pairs
  // outermost (a wave of CTAs sweeps every column tile of B), 1 = column
  // tiles outermost (a wave reuses each B column tile across all row pairs),
  // 2 = groups of row pairs, each swept with column tiles outermost
  int col_major;
  // experts whose rows (weight gradients: reduction rows) lie outside
  // [row_min, row_max) own no units in this launch (row_max 0: no bound);
  // set by launch_grouped_gemm when it splits a launch
  int row_min;
  int row_max;
  // kWgrad: 1 = add the result to the bf16 values already in `out` (one
  // rounding of old + new); experts with no rows leave theirs untouched
  int accumulate;
  // kFc2 / kDgrad: 1 = tmC maps `out` as [M_cap, N] bf16 (ldo == N), box 32
  // columns x 32 rows with 64-byte swizzle, and the epilogue writes whole
  // 32-row groups of a tile with staged TMA stores (a ragged last group of
  // an expert with plain stores); 0 = plain stores throughout.  kFc1Act
  // (bf16 outputs): the same for H (out2, tmC) and A (out, tmD)
  int tma_out;
  // gathered operand (the permute fused into the operand load): the
  // operand's expert-major row r is row gather_pair[r] / gather_k of the
  // token tensor gather_src [gather_T, gather_ld] (zeros for pad rows,
  // gather_pair[r] < 0).  The ragged-row kinds gather their K-major A (tmA
  // unused); kWgrad gathers the reduction rows of A (gather_operand 0, tmA
  // unused) or of B (1, tmB unused).  NULL: no gather.
  const int32_t* gather_pair;
  int gather_k;
  int gather_T;
  int gather_operand;
  const uint16_t* gather_src;
  long long gather_ld;
};

// Launches the persistent grouped GEMM of `kind` (act: MOE_ACT_*) on `s`.
// tc: the output's tensor map for kWgrad ([E, R, N] bf16, see wgrad_skinny
// for its box), and with tma_out for kFc2 / kDgrad (out) and kFc1Act (H,
// out2); td: with tma_out, kFc1Act's A (out) and kDgradAct's A' (out3);
// for kWgrad of a skinny layer, optionally the output map with the
// large-expert box (32 columns).  The [rows, cols] maps of tma_out have
// 32 x 32 boxes with 64-byte swizzle.  Unused maps may be any valid map (td
// defaults to tc).
// A layer whose experts average fewer than kPairRows rows runs the
// single-CTA configuration (weight gradients: the skinny one, see
// wgrad_skinny); in automatic pair mode its experts that do reach kPairRows
// rows run first, in a launch of their own with the pair configuration
// (weight gradients: the large-expert one when td is given).  *launched:
// the number of kernels launched (1 or 2).
cudaError_t launch_grouped_gemm(GemmKind kind, int act, const CUtensorMap& ta,
                                const CUtensorMap& tb, const CUtensorMap& tc,
                                const GemmArgs& args, int num_sms, cudaStream_t s,
                                bool mx = false, const CUtensorMap* td = nullptr,
                                int* launched = nullptr);

// Weight gradients use the skinny-expert configuration when the average
// rows per expert (M_cap / E, known on the host without reading counts) is
// below kSkinnyRows; its output tensor map box is then 64 x 32 (128-byte
// swizzle), else 32 x 32 (64-byte swizzle).
constexpr int kSkinnyRows = 512;
bool wgrad_skinny(const GemmArgs& g);

// Pair mode (2-SM MMAs over 256-row units) for the ragged-row kinds:
// kPairAuto uses it when the average rows per expert (M_cap / E, known on
// the host) reach kPairRows; kPairNever / kPairAlways force the choice (for
// measurement and tests).  set_pair_mode returns the previous mode, or -1
// for an unknown one.
constexpr int kPairNever = 0, kPairAuto = 1, kPairAlways = 2;
constexpr int kPairRows = 256;
int set_pair_mode(int mode);
int pair_mode();
bool use_pair(GemmKind kind, const GemmArgs& g);

// The activation and its derivative as separate memory passes (act.cu):
// A = act(H) and dH = act'(H; dA) over the rows below offsets[E] (at most
// rows_cap); H is [rows, n1], A / dA are [rows, n].
cudaError_t launch_act_fwd(const uint16_t* h, const int32_t* offsets, int E, long long rows_cap,
                           int n, int act, uint16_t* a, int num_sms, cudaStream_t st);
cudaError_t launch_act_bwd(const uint16_t* h, const uint16_t* da, const int32_t* offsets, int E,
                           long long rows_cap, int n, int act, uint16_t* dh, int num_sms,
                           cudaStream_t st);

// Box shapes (elements) the kernels expect for each operand's tensor map.
constexpr int kBM = 128, kBN = 256, kBK = 64;

}  // namespace moe
