// mxgemm.cuh - host-side interface of the MXFP8 kernels: the block-scaled
// grouped GEMM (mx.cu) and the quantisers (mx_quant.cu).
//
// Scale layouts read by the block-scaled GEMM.  All are made of 512-byte
// chunks in the order tcgen05.cp moves them into TMEM (128 operand rows x 4
// consecutive 32-blocks of the reduction index; byte mx_chunk_off(r, b), see
// mx.cuh).  Which 128 rows and which 4 blocks a chunk holds depends on the
// operand:
//   row tiles     - an activation [rows, K] with blocks along K, read in
//                   128-row tiles that start at offsets[e] + 128 i: chunk
//                   (row0 / 32) * (K / 128) + k / 128.  Size rows * K / 8.
//   weight tiles  - a weight viewed as [rows, K] (rows = E * N) with blocks
//                   along K, read in 128-row tiles from row 0: chunk
//                   (row / 128) * (K / 128) + k / 128.  Size rows * K / 32.
//   K tiles       - a transposed copy [C, M] with blocks of 32 rows of one
//                   expert, read by the weight gradient in reduction steps
//                   of 128 rows that start at offsets[e] + 128 i: chunk
//                   (k0 / 32) * (C / 128) + c / 128.  Size M * C / 8.
//   W2 column tiles (forward FC2, moe_mx_quantize_weights) - see moe.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

enum class MxKind : int {
  kFc2 = 0,       // Y = A W2: A row tiles, W2 [E, K, N] N-major with column tiles
  kDgrad = 1,     // out = G W^T: G row tiles, W [E*N, K] K-major with weight tiles
  kDgradAct = 2,  // as kDgrad, then dH = act'(H; .) in the epilogue
  kWgrad = 3,     // dW_e = P_e^T Q_e from transposed copies [R, M], [N, M] (K tiles)
};

struct MxGemmArgs {
  const int32_t* offsets;  // [E+1], multiples of 32
  int E;
  int M_cap;
  int K;                   // reduction length of the ragged-row kinds (multiple of 128)
  int N;                   // accumulator columns (multiple of 128)
  int R;                   // kWgrad: output rows per expert (multiple of 128)
  const uint8_t* a_s;      // A scales
  const uint8_t* b_s;      // B scales
  long long a_s_bytes;     // sizes of the two scale buffers (pair mode loads their
  long long b_s_bytes;     // chunks with TMA; 0: pair mode is not used)
  uint16_t* out;           // ragged-row kinds: [M_cap, ldo] bf16
  long long ldo;
  const uint16_t* aux;     // kDgradAct: H [M_cap, ld_aux]
  long long ld_aux;
  // kFc2 / kDgrad, optional (q_out == nullptr: none): row-wise MXFP8 copy of
  // the bf16 output - codes [M_cap, N], plain E8M0 scales [M_cap, N/32]
  uint8_t* q_out;
  uint8_t* s_out;
  int32_t* err;
  // kFc2 / kDgrad without q_out: 1 = tmC maps `out` as [M_cap, N] bf16
  // (ldo == N), box 32 columns x 32 rows with 64-byte swizzle, and the
  // epilogue writes whole 32-row groups with staged TMA stores; 0 = plain
  // stores
  int tma_out;
  // kWgrad: experts whose reduction rows lie outside [row_min, row_max) own
  // no units in this launch (row_max 0: no bound); set by launch_mx_gemm
  // when it splits a launch
  int row_min;
  int row_max;
  // also: the tma_out staged stores of kDgradAct's bf16 dH when dh_q is set
  // kDgradAct, optional (dh_q == nullptr: none): GroupGemm + dActivation +
  // Quantize/Transpose - the epilogue also writes the MXFP8 copies of the
  // bf16 dH it stores, as the tiled activation quantiser would: row-wise
  // codes dh_q [M_cap, n1] with scales dh_s in row tiles (FC1-dgrad's A),
  // and the transposed copy dh_qT [n1, M_cap] with scales dh_sT in K tiles
  // (FC1-wgrad's B)
  uint8_t* dh_q;
  uint8_t* dh_s;
  uint8_t* dh_qT;
  uint8_t* dh_sT;
  int n1;
  // kWgrad: 1 = add the result to the bf16 values already in `out` ([E, R,
  // N], one rounding of old + new); experts with no rows leave theirs
  // untouched
  int accumulate;
};

// W2 [E, n, d]: blocks of 32 rows per column (q, s: column tiles as in
// moe.h); with q_rows also blocks of 32 columns per row (q_rows, s_rows in
// weight tiles of W2 viewed as [E*n, d]) from the same read; offsets (may
// be null): experts with no rows are skipped and left untouched
cudaError_t launch_mx_quantize_weights(const uint16_t* w2, int E, int n, int d,
                                       const int32_t* offsets, uint8_t* q, uint8_t* s,
                                       uint8_t* q_rows, uint8_t* s_rows, int num_sms,
                                       cudaStream_t st);
// ragged activation: row-wise codes q / scales s (q may be null: transposed
// copy only) and the transposed copy qT / sT (may be null).  tiled = false:
// plain scales s [rows, cols/32], sT [cols, rows/32]; tiled = true (cols a
// multiple of 128, else cudaErrorInvalidValue): s in row tiles, sT in K
// tiles.
cudaError_t launch_mx_quantize_act(const uint16_t* src, int rows, int cols, const int32_t* offsets,
                                   int E, uint8_t* q, uint8_t* s, uint8_t* qT, uint8_t* sT,
                                   int32_t* err, bool tiled, int num_sms, cudaStream_t st);
// [rows, cols] (rows a multiple of 128) with blocks along cols, weight tiles;
// offsets (may be null): expert e holds rows [e, e+1) * rows_per_e (a
// multiple of 128) and is skipped, untouched, when it has no rows
cudaError_t launch_mx_quantize_rows_w(const uint16_t* src, long long rows, int cols,
                                      const int32_t* offsets, long long rows_per_e, uint8_t* q,
                                      uint8_t* s, int num_sms, cudaStream_t st);
// plain transposed scales sT [cols, rows/32] -> K tiles
cudaError_t launch_mx_retile_t(const uint8_t* sT, int rows, int cols, const int32_t* offsets,
                               int E, uint8_t* out, int num_sms, cudaStream_t st);
// tc: output map of kWgrad ([E, R, N] bf16, box 64 x 32, 128-byte swizzle)
// A weight gradient of a layer below kPairRows rows per expert runs its
// experts of kPairRows reduction rows or more first, in a launch of their
// own with 2-SM tiles (automatic pair mode); *launched: kernels launched.
cudaError_t launch_mx_gemm(MxKind kind, int act, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const MxGemmArgs& g, int num_sms,
                           cudaStream_t st, int* launched = nullptr);

}  // namespace moe
