// mx.cu - MXFP8 kernels:
//   * mx_quantize_weights: W2 [E, n, d] bf16 -> E4M3 codes [E, n, d] and
//     E8M0 scales over 32 consecutive rows (FC2's reduction index) per
//     column, in the MMA-tiled layout (see mx.cuh).
//   * mx_quantize_rows_w: any weight viewed as [rows, K] with blocks along
//     K (the reduction index of a data gradient), scales in weight tiles.
//   * mx_quantize_act: group-aware quantiser of a ragged [rows, cols]
//     activation: row-wise 1x32 blocks, plus the transposed copy with
//     column-wise 32x1 blocks that never cross an expert's rows; scales
//     plain or in the tiles the GEMM reads (see mxgemm.cuh).
//   * mx_retile_t: plain transposed scales -> the weight gradient's K tiles.
//   * mx_gemm: block-scaled MXFP8 grouped GEMM
//     (tcgen05.mma.kind::mxf8f6f4.block_scale) for FC2, the two data
//     gradients (FC2's with the dActivation epilogue) and the ragged-K
//     weight gradients; same persistent warp-specialised structure as the
//     bf16 grouped GEMM.
// [CuTe] "무엇을 해결하려는가" and "핵심 아이디어": MXFP8 output and transposed
// output; [TE] "Transformer Engine이 제공하는 세 가지 구성 요소": group-aware
// MXFP8 quantisation and an MXFP8 grouped GEMM; [TE] "다음 단계: NVFP4, GEMM
// 융합 양자화, A2A 오버랩": the backward's GroupGemm + dActivation +
// Quantize/Transpose.
#include <cuda_runtime.h>

#include "act.cuh"
#include "mx.cuh"
#include "mxgemm.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- weights
// With the routing offsets given, an expert that holds no rows is skipped:
// no GEMM reads its weights (its row tiles do not exist), so its codes and
// scales are left as they were.  Each block first lists the used experts in
// order (one warp, 32 experts a ballot) and the grid-stride loop then runs
// over the used experts' work alone, as densely as over all experts.
// Without offsets the list is the identity over n_all experts.  Every
// thread of the block must call it (one barrier).
__device__ __forceinline__ int used_experts(const int32_t* __restrict__ offsets, int n_all,
                                            int* s_list, int* s_count) {
  if (offsets == nullptr) return n_all;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int cnt = 0;
    for (int base = 0; base < n_all; base += 32) {
      const int e = base + lane;
      const bool used = e < n_all && __ldg(offsets + e + 1) != __ldg(offsets + e);
      const uint32_t m = __ballot_sync(0xffffffffu, used);
      if (used) s_list[cnt + __popc(m & ((1u << lane) - 1u))] = e;
      cnt += __popc(m);
    }
    if (lane == 0) *s_count = cnt;
  }
  __syncthreads();
  return *s_count;
}

// W2 [E, n, d] quantised for the forward FC2 alone: blocks of 32 rows (FC2's
// reduction index n) per column.  One thread: 8 consecutive columns x one
// 32-row block of one expert (a warp reads 512 contiguous bytes per row).
__global__ void __launch_bounds__(256)
    mx_quantize_weights_kernel(const uint4* __restrict__ w, int E, int n, int d,
                               const int32_t* __restrict__ offsets, uint2* __restrict__ q,
                               uint8_t* __restrict__ s) {
  __shared__ int s_list[MOE_MAX_EXPERTS];
  __shared__ int s_count;
  const int ne = used_experts(offsets, E, s_list, &s_count);
  const int d8 = d / 8;
  const long long total = static_cast<long long>(ne) * (n / 32) * d8;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(g % d8);
    const long long eb = g / d8;
    const int b = static_cast<int>(eb % (n / 32));
    const int eu = static_cast<int>(eb / (n / 32));
    const int e = offsets ? s_list[eu] : eu;
    const long long row0 = static_cast<long long>(e) * n + 32LL * b;
    float v[32][8];
    float amax[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint4 x = __ldg(w + (row0 + i) * d8 + c8);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[i][2 * j] = bf16_lo(xw[j]);
        v[i][2 * j + 1] = bf16_hi(xw[j]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) amax[j] = fmaxf(amax[j], fabsf(v[i][j]));
    }
    uint32_t code[8];
    float inv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      code[j] = mx_scale_code(amax[j]);
      inv[j] = mx_inv_scale(code[j]);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t w0 = e4m3x2(v[i][0] * inv[0], v[i][1] * inv[1]) |
                          (e4m3x2(v[i][2] * inv[2], v[i][3] * inv[3]) << 16);
      const uint32_t w1 = e4m3x2(v[i][4] * inv[4], v[i][5] * inv[5]) |
                          (e4m3x2(v[i][6] * inv[6], v[i][7] * inv[7]) << 16);
      q[(row0 + i) * d8 + c8] = make_uint2(w0, w1);
    }
    // scales: chunk (b/4, c/128) of expert e
    uint8_t* se = s + static_cast<long long>(e) * (n / 32) * d;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c8 * 8 + j;
      const long long chunk = static_cast<long long>(b / 4) * (d / 128) + c / 128;
      se[chunk * 512 + mx_chunk_off(c & 127, b & 3)] = static_cast<uint8_t>(code[j]);
    }
  }
}

// W2 [E, n, d] quantised for both FC2 (blocks of 32 rows along its
// reduction index n, per column) and FC2-dgrad (blocks of 32 columns along
// its reduction index d, per row), so that MXFP8 training takes both copies
// from one read of W2.
// A warp covers one 32-row block x 128 columns: lane = 16 * half + i holds
// rows 16 * half .. +15 of columns 8 * i .. +7 (values kept as packed bf16
// pairs).  A column's 32-row maximum combines the two halves (lanes 16
// apart); a row's 32-column maximum combines four adjacent lanes.
__global__ void __launch_bounds__(256)
    mx_quantize_w2_kernel(const uint4* __restrict__ w, int E, int n, int d,
                          const int32_t* __restrict__ offsets,
                          uint2* __restrict__ q, uint8_t* __restrict__ s,
                          uint2* __restrict__ qr, uint8_t* __restrict__ sr) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int d8 = d / 8;
  __shared__ int s_list[MOE_MAX_EXPERTS];
  __shared__ int s_count;
  const int ne = used_experts(offsets, E, s_list, &s_count);
  const int cw = d / 128;                                  // warps per 32-row block
  const long long nwarps = static_cast<long long>(ne) * (n / 32) * cw;
  for (long long wi = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) / 32;
       wi < nwarps; wi += static_cast<long long>(gridDim.x) * blockDim.x / 32) {
    const int c8 = static_cast<int>(wi % cw) * 16 + (lane & 15);
    const long long eb = wi / cw;
    const int b = static_cast<int>(eb % (n / 32));
    const int eu = static_cast<int>(eb / (n / 32));
    const int e = offsets ? s_list[eu] : eu;
    const long long row0 = static_cast<long long>(e) * n + 32LL * b + 16 * half;
    uint32_t x[16][4];
    float amax[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint4 v = __ldg(w + (row0 + i) * d8 + c8);
      x[i][0] = v.x; x[i][1] = v.y; x[i][2] = v.z; x[i][3] = v.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        amax[2 * j] = fmaxf(amax[2 * j], fabsf(bf16_lo(x[i][j])));
        amax[2 * j + 1] = fmaxf(amax[2 * j + 1], fabsf(bf16_hi(x[i][j])));
      }
    }
    uint32_t code[8];
    float inv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], 16));
      code[j] = mx_scale_code(amax[j]);
      inv[j] = mx_inv_scale(code[j]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w0 = e4m3x2(bf16_lo(x[i][0]) * inv[0], bf16_hi(x[i][0]) * inv[1]) |
                          (e4m3x2(bf16_lo(x[i][1]) * inv[2], bf16_hi(x[i][1]) * inv[3]) << 16);
      const uint32_t w1 = e4m3x2(bf16_lo(x[i][2]) * inv[4], bf16_hi(x[i][2]) * inv[5]) |
                          (e4m3x2(bf16_lo(x[i][3]) * inv[6], bf16_hi(x[i][3]) * inv[7]) << 16);
      q[(row0 + i) * d8 + c8] = make_uint2(w0, w1);
    }
    {   // column scales, chunk (b/4, c/128) of expert e: both halves hold the
        // same codes, half 0 stores columns 8i..8i+3 and half 1 8i+4..8i+7
        // (each store then touches the chunk's 4 lines once per warp)
      uint8_t* se = s + static_cast<long long>(e) * (n / 32) * d;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int c = c8 * 8 + jj + 4 * half;
        const long long chunk = static_cast<long long>(b / 4) * (d / 128) + c / 128;
        se[chunk * 512 + mx_chunk_off(c & 127, b & 3)] =
            static_cast<uint8_t>(half ? code[jj + 4] : code[jj]);
      }
    }
    {
      const int c = c8 * 8;                     // first column of this lane
      // the 4 block scales of row 16 * half + l end in lane 16 * half + l
      // (gathered by shuffles), stored as one 4-byte word per row
      uint32_t my_row_sc = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(x[i][j])), fabsf(bf16_hi(x[i][j]))));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const uint32_t sc = mx_scale_code(m);
        const float iv = mx_inv_scale(sc);
        const uint32_t w0 = e4m3x2(bf16_lo(x[i][0]) * iv, bf16_hi(x[i][0]) * iv) |
                            (e4m3x2(bf16_lo(x[i][1]) * iv, bf16_hi(x[i][1]) * iv) << 16);
        const uint32_t w1 = e4m3x2(bf16_lo(x[i][2]) * iv, bf16_hi(x[i][2]) * iv) |
                            (e4m3x2(bf16_lo(x[i][3]) * iv, bf16_hi(x[i][3]) * iv) << 16);
        const long long r = row0 + i;
        qr[r * d8 + c8] = make_uint2(w0, w1);
        // lanes 16 * half + 4 cb hold this row's scale of column block cb
        uint32_t packed = 0;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
          packed |= __shfl_sync(0xffffffffu, sc, (lane & 16) + 4 * cb) << (8 * cb);
        if ((lane & 15) == i) my_row_sc = packed;
      }
      // weight tiles of W2 viewed as [E*n, d]: row r's 4 bytes are
      // contiguous in its chunk (the 4 column blocks of c / 128)
      const long long r = row0 + (lane & 15);
      const long long chunk = (r / 128) * (d / 128) + c / 128;
      *reinterpret_cast<uint32_t*>(sr + chunk * 512 + mx_chunk_off(static_cast<int>(r & 127), 0)) =
          my_row_sc;
    }
  }
}

// ---------------------------------------------------------------- activations
// expert holding row `row` (offsets in shared memory): the last e with
// s_off[e] <= row; empty experts share their start with the next one, so
// the last such e is the one whose range contains the row
__device__ __forceinline__ int expert_of_row(const int* s_off, int E, int row) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_off[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// start of the 128-row tile (or weight-gradient reduction step) that holds
// the 32-row block starting at row r32: tiles start at offsets[e] + 128 i.
// Clamped so that a malformed offsets array (reported separately) still
// gives an index inside the buffer.
__device__ __forceinline__ int tile_start(const int* s_off, int E, int r32) {
  const int e = expert_of_row(s_off, E, r32);
  const int oe = min(max(s_off[e], 0), r32) & ~31;
  return oe + ((r32 - oe) & ~127);
}

// Plain scale layouts (s [rows, cols/32], sT [cols, rows/32]), any width
// that is a multiple of 32: one warp takes a 32-row block (inside one
// expert) x a 32-column block, lane = row.
__global__ void __launch_bounds__(256)
    mx_quantize_act_kernel(const uint4* __restrict__ src, int rows, int cols,
                           const int32_t* __restrict__ offsets, int E,
                           uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                           uint8_t* __restrict__ qT, uint8_t* __restrict__ sT,
                           int32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int cb_n = cols / 32;
  const long long nwarps = static_cast<long long>(rows / 32) * cb_n;
  const int used = min(max(offsets[E], 0), rows);
  // a 32-row block must lie inside one expert: expert starts must be
  // multiples of 32 (reported, not repaired)
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x)
      if (offsets[e] & 31) set_err(err, MOE_DEV_BAD_OFFSETS);
  for (long long wi = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) / 32;
       wi < nwarps; wi += static_cast<long long>(gridDim.x) * blockDim.x / 32) {
    const int rb = static_cast<int>(wi / cb_n);
    const int cb = static_cast<int>(wi % cb_n);
    const int r = rb * 32 + lane;
    if (rb * 32 >= used) continue;       // rows past every expert: untouched
    float v[32];
    const uint4* p = src + (static_cast<long long>(r) * cols + cb * 32) / 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 x = __ldg(p + k);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * k + 2 * j] = bf16_lo(xw[j]);
        v[8 * k + 2 * j + 1] = bf16_hi(xw[j]);
      }
    }
    if (q) {
      uint32_t qw[8];
      const uint32_t sc = mx_quant32(v, qw);
      uint4* qo = reinterpret_cast<uint4*>(q + static_cast<long long>(r) * cols + cb * 32);
      qo[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      qo[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
      s[static_cast<long long>(r) * cb_n + cb] = static_cast<uint8_t>(sc);
    }
    if (qT) {
      uint32_t my_sc = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        uint32_t code;
        const uint32_t scj = mx_quant_lanes(v[j], code);
        qT[static_cast<long long>(cb * 32 + j) * rows + r] = static_cast<uint8_t>(code);
        if (lane == j) my_sc = scj;
      }
      const int c = cb * 32 + lane;
      sT[static_cast<long long>(c) * (rows / 32) + rb] = static_cast<uint8_t>(my_sc);
    }
  }
}

// Tiled copies for widths that are multiples of 128 (the GEMMs' layouts):
// one warp takes a 32-row block (inside one expert) x 128 columns, lane
// 16 * half + i holding rows 16 * half .. +15 of columns 8 i .. 8 i + 7 as
// packed bf16 pairs (the two-direction W2 quantiser's arrangement).  A
// column's 32-row maximum combines the two halves (lanes 16 apart) and a
// row's 32-column maximum four adjacent lanes.  The transposed codes of a
// column then leave as one 16-byte store per lane (16 consecutive rows of
// qT's row), the row-wise codes as one 8-byte store per row and lane, the
// row scales as one 4-byte word per row (the four blocks of a 128-column
// chunk are adjacent in its row tile), and the column scales as bytes split
// across both halves, which hold the same codes.  The one-block-per-warp
// kernel above spends most of its instructions on 32 single-byte stores
// and 32 warp reductions per block for the transposed copy (848 warp
// instructions per 32 x 32 block under ncu on a 8,192 x 8,192 dY).
__global__ void __launch_bounds__(256)
    mx_quantize_act_w_kernel(const uint4* __restrict__ src, int rows, int cols,
                             const int32_t* __restrict__ offsets, int E,
                             uint2* __restrict__ q, uint8_t* __restrict__ s,
                             uint8_t* __restrict__ qT, uint8_t* __restrict__ sT,
                             int32_t* __restrict__ err) {
  __shared__ int s_off[MOE_MAX_EXPERTS + 1];
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int li = lane & 15;
  const int cw = cols / 128;
  const int c8n = cols / 8;
  const long long nwarps = static_cast<long long>(rows / 32) * cw;
  const int used = min(max(offsets[E], 0), rows);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = offsets[e];
  __syncthreads();
  // a 32-row block must lie inside one expert (reported, not repaired)
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e <= E; e += blockDim.x)
      if (offsets[e] & 31) set_err(err, MOE_DEV_BAD_OFFSETS);
  for (long long wi = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) / 32;
       wi < nwarps; wi += static_cast<long long>(gridDim.x) * blockDim.x / 32) {
    const int rb = static_cast<int>(wi / cw);
    const int cc = static_cast<int>(wi - static_cast<long long>(rb) * cw);
    if (rb * 32 >= used) continue;       // rows past every expert: untouched
    const int c8 = cc * 16 + li;
    const int row0 = rb * 32 + 16 * half;
    uint32_t x[16][4];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 v = __ldg(src + static_cast<long long>(row0 + k) * c8n + c8);
      x[k][0] = v.x; x[k][1] = v.y; x[k][2] = v.z; x[k][3] = v.w;
    }
    const int t0 = tile_start(s_off, E, rb * 32);
    const long long chunk = static_cast<long long>(t0 / 32) * cw + cc;
    if (qT) {
      float amax[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int k = 0; k < 16; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax[2 * j] = fmaxf(amax[2 * j], fabsf(bf16_lo(x[k][j])));
          amax[2 * j + 1] = fmaxf(amax[2 * j + 1], fabsf(bf16_hi(x[k][j])));
        }
      uint32_t code[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], 16));
        code[j] = mx_scale_code(amax[j]);
        const float inv = mx_inv_scale(code[j]);
        // column 8 li + j, rows row0 .. row0 + 15: 16 bytes of qT's row
        auto val = [&](int k) {
          return (j & 1) ? bf16_hi(x[k][j >> 1]) : bf16_lo(x[k][j >> 1]);
        };
        uint32_t w[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          w[m] = e4m3x2(val(4 * m) * inv, val(4 * m + 1) * inv) |
                 (e4m3x2(val(4 * m + 2) * inv, val(4 * m + 3) * inv) << 16);
        const long long c = static_cast<long long>(cc) * 128 + 8 * li + j;
        *reinterpret_cast<uint4*>(qT + c * rows + row0) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      // column scales in the K tile of this row block: half 0 stores
      // columns 8 li .. +3, half 1 8 li + 4 .. +7
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = jj + 4 * half;
        sT[chunk * 512 + mx_chunk_off(8 * li + j, (rb * 32 - t0) >> 5)] =
            static_cast<uint8_t>(half ? code[jj + 4] : code[jj]);
      }
    }
    if (q) {
      // the 4 block scales of row 16 * half + l end in lane 16 * half + l
      // (gathered by shuffles) and are stored as one word
      uint32_t my_row_sc = 0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m = fmaxf(m, fmaxf(fabsf(bf16_lo(x[k][j])), fabsf(bf16_hi(x[k][j]))));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const uint32_t sc = mx_scale_code(m);
        const float iv = mx_inv_scale(sc);
        const uint32_t w0 = e4m3x2(bf16_lo(x[k][0]) * iv, bf16_hi(x[k][0]) * iv) |
                            (e4m3x2(bf16_lo(x[k][1]) * iv, bf16_hi(x[k][1]) * iv) << 16);
        const uint32_t w1 = e4m3x2(bf16_lo(x[k][2]) * iv, bf16_hi(x[k][2]) * iv) |
                            (e4m3x2(bf16_lo(x[k][3]) * iv, bf16_hi(x[k][3]) * iv) << 16);
        q[static_cast<long long>(row0 + k) * c8n + c8] = make_uint2(w0, w1);
        uint32_t packed = 0;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb)
          packed |= __shfl_sync(0xffffffffu, sc, (lane & 16) + 4 * cb) << (8 * cb);
        if (li == k) my_row_sc = packed;
      }
      *reinterpret_cast<uint32_t*>(s + chunk * 512 + mx_chunk_off(row0 + li - t0, 0)) = my_row_sc;
    }
  }
}

// ---------------------------------------------------------------- row-wise weights
// [rows, cols] with blocks of 32 along cols, scales in weight tiles (128-row
// tiles from row 0).  A warp takes 32 consecutive blocks (2 KB, contiguous
// since cols is a multiple of 128): in its k-th load lane l reads 16-byte
// piece 32k + l, so each load instruction covers 512 contiguous bytes; lane
// l then holds a quarter (8 values) of blocks 8k + l/4, and a block's
// maximum takes two shuffles across its 4 lanes.
// With offsets, rows_per_e (a multiple of 128) rows make one expert: an
// expert then starts at a block index that is a multiple of 512, so a warp's
// 32 blocks and a 128-row scale tile never straddle two experts.
__global__ void __launch_bounds__(256)
    mx_quantize_rows_w_kernel(const uint4* __restrict__ src, long long rows, int cols,
                              const int32_t* __restrict__ offsets, long long rows_per_e,
                              uint2* __restrict__ q, uint8_t* __restrict__ s) {
  __shared__ int s_list[MOE_MAX_EXPERTS];
  __shared__ int s_count;
  const int lane = threadIdx.x & 31;
  const int cb_n = cols / 32;
  const int ne = used_experts(offsets, static_cast<int>(rows / rows_per_e), s_list, &s_count);
  const long long warps_e = rows_per_e * cb_n / 32;  // cols / 32 is a multiple of 4; see the launch
  const long long nwarps = ne * warps_e;
  for (long long wi = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) / 32;
       wi < nwarps; wi += static_cast<long long>(gridDim.x) * blockDim.x / 32) {
    const long long eu = wi / warps_e;
    const long long e = offsets ? s_list[eu] : eu;
    const long long g0 = (e * warps_e + (wi - eu * warps_e)) * 32;   // first block of the warp
    uint32_t x[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(src + g0 * 4 + 32 * k + lane);
      x[k][0] = v.x; x[k][1] = v.y; x[k][2] = v.z; x[k][3] = v.w;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(x[k][j])), fabsf(bf16_hi(x[k][j]))));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const uint32_t sc = mx_scale_code(m);
      const float iv = mx_inv_scale(sc);
      const uint32_t w0 = e4m3x2(bf16_lo(x[k][0]) * iv, bf16_hi(x[k][0]) * iv) |
                          (e4m3x2(bf16_lo(x[k][1]) * iv, bf16_hi(x[k][1]) * iv) << 16);
      const uint32_t w1 = e4m3x2(bf16_lo(x[k][2]) * iv, bf16_hi(x[k][2]) * iv) |
                          (e4m3x2(bf16_lo(x[k][3]) * iv, bf16_hi(x[k][3]) * iv) << 16);
      q[g0 * 4 + 32 * k + lane] = make_uint2(w0, w1);  // 8 codes: 256 contiguous bytes a warp
      if ((lane & 3) == 0) {
        const long long g = g0 + 8 * k + lane / 4;       // this block
        const long long r = g / cb_n;
        const int cb = static_cast<int>(g - r * cb_n);
        const long long chunk = (r / 128) * (cols / 128) + cb / 4;
        s[chunk * 512 + mx_chunk_off(static_cast<int>(r & 127), cb & 3)] = static_cast<uint8_t>(sc);
      }
    }
  }
}

// ---------------------------------------------------------------- scale re-tiling
// plain transposed scales sT [cols, rows/32] -> K tiles (one thread a byte)
__global__ void __launch_bounds__(256)
    mx_retile_t_kernel(const uint8_t* __restrict__ sT, int rows, int cols,
                       const int32_t* __restrict__ offsets, int E, uint8_t* __restrict__ out) {
  __shared__ int s_off[MOE_MAX_EXPERTS + 1];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = offsets[e];
  __syncthreads();
  const int rb_n = rows / 32;
  const int used = min(max(s_off[E], 0), rows);
  const long long total = static_cast<long long>(cols) * rb_n;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(g / rb_n);
    const int rb = static_cast<int>(g - static_cast<long long>(c) * rb_n);
    if (rb * 32 >= used) continue;
    const int t0 = tile_start(s_off, E, rb * 32);
    const long long chunk = static_cast<long long>(t0 / 32) * (cols / 128) + c / 128;
    out[chunk * 512 + mx_chunk_off(c & 127, (rb * 32 - t0) >> 5)] = sT[g];
  }
}

// ---------------------------------------------------------------- block-scaled GEMM
// Output tiles are 128 x 256, computed as two 128 x 128 block-scaled MMAs per
// 32-element step of K (each half with its own B scale chunk).  A pipeline
// stage holds one 128-byte swizzle atom of K (128 FP8 elements) of A and of
// both B halves plus their three scale chunks: 48 KB of operands for 8.4
// MFLOP, the same bytes-per-FLOP as the bf16 kernel's 128 x 256 x 64 stage
// at twice the tensor rate.
constexpr int QBM = 128, QBN = 256, QHN = 128;   // tile rows, tile columns, MMA N
constexpr int QBK = 128;                          // FP8 elements (= bytes) of K per stage
constexpr int QA_BYTES = QBM * QBK;               // 16 KB
constexpr int QBH_BYTES = QHN * QBK;              // 16 KB per B half
constexpr int QSF_OFF = QA_BYTES + 2 * QBH_BYTES; // scale chunks: SFA, SFB half 0, SFB half 1
constexpr int QSTAGE_BYTES = QSF_OFF + 2048;      // 50 KB (stages stay 1024-byte aligned)
constexpr int QTHREADS = 320;
constexpr int QEPI_WARPS = 8;
constexpr int QTMEM_COLS = 512;
constexpr int QSF_TMEM = QBN;                     // scale columns after the accumulator
constexpr int QSF_COLS = 12;                      // a stage's three chunks, 4 columns each
constexpr int QBOX_BYTES = 32 * 64 * 2;           // staged output box: 32 rows x 64 bf16

// TMEM holds one 256-column accumulator (the scale columns leave no room
// for a second); the epilogue moves it to registers and releases it at once,
// so the next tile's MMAs overlap the conversion and stores.  The weight
// gradient stages its output for TMA stores (one box per epilogue warp plus
// a box of zeros for experts with no rows) and keeps three stages; the other
// kinds keep four.
template <MxKind KIND>
struct QCfg {
  static constexpr bool W = (KIND == MxKind::kWgrad);
  static constexpr int stages = W ? 3 : 4;
  static constexpr int stg_bytes = W ? (QEPI_WARPS + 1) * QBOX_BYTES : 0;
};
template <MxKind KIND>
constexpr size_t mx_smem_bytes(int E) {
  return 1024 + static_cast<size_t>(QCfg<KIND>::stages) * QSTAGE_BYTES + QCfg<KIND>::stg_bytes +
         (2 * QCfg<KIND>::stages + 4) * 8 + 16 + 2 * (E + 1) * 4;
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: A/B E4M3 (format 0),
// bit 15/16 A/B major, bits 17-22 N>>3, bit 23 scale type (1 = E8M0),
// bits 24-28 M>>4; scale-factor byte selectors: B bits 4-5, A bits 29-30.
constexpr uint32_t idesc_mx(int M, int N, bool a_mn, bool b_mn) {
  return ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// no-swizzle descriptor of a 512-byte scale chunk (32 rows x 16 bytes,
// 8-row core matrices 128 bytes apart)
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(512 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

struct QTile {
  int e;
  int row0, rows;   // ragged-row kinds: first global row, valid rows
  int m0;           // kWgrad: first output row within the expert
  int n0;           // first accumulator column
  int nh;           // 128-column halves of the tile inside N (1 or 2)
  int kblocks;      // QBK-element reduction steps
  int k0;           // kWgrad: first reduction row (global)
  int klast;        // kWgrad: valid rows of the last step (a multiple of 32)
  bool mc;          // the pair shares (multicasts) this B block
  bool ghost;       // no output: past the expert's row blocks, or past N
};

// Work units of a 2-CTA cluster.  With at least two 128-row blocks, a unit
// is two consecutive row blocks that share one 256-column block of B (CTA r
// takes row block 2i + r; each CTA fetches one 128-column half of B and
// multicasts it into both).  An expert with a single row block pairs along
// N instead: CTA r takes column block 2i + r and loads its own operands.  A
// CTA whose row or column block lies past the expert or past N is a ghost:
// it still fetches and multicasts its half of a shared B block, and still
// frees each stage in both CTAs, but loads, computes and stores nothing
// else.
constexpr int QCL = 2;
constexpr uint16_t kQPair = 0x3;
template <MxKind KIND>
__device__ __forceinline__ int mx_row_blocks(const MxGemmArgs& g, const int* s_off, int e) {
  return (KIND == MxKind::kWgrad) ? g.R / QBM : (s_off[e + 1] - s_off[e] + QBM - 1) / QBM;
}

template <MxKind KIND>
__device__ __forceinline__ int mx_tiles_of_expert(const MxGemmArgs& g, const int* s_off, int e) {
  const int nt = (g.N + QBN - 1) / QBN;
  const int mt = mx_row_blocks<KIND>(g, s_off, e);
  if (mt == 1) return (nt + 1) / 2;
  return ((mt + 1) / 2) * nt;
}

template <MxKind KIND>
__device__ __forceinline__ QTile mx_decode(const MxGemmArgs& g, const int* s_off, const int* s_ts,
                                           int t, int rank) {
  int lo = 0, hi = g.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_ts[mid + 1] <= t) lo = mid + 1;
    else hi = mid;
  }
  const int nt = (g.N + QBN - 1) / QBN;
  const int local = t - s_ts[lo];
  const int mt = mx_row_blocks<KIND>(g, s_off, lo);
  QTile tl;
  tl.e = lo;
  int mi;
  if (mt == 1) {
    tl.mc = false;
    mi = 0;
    tl.n0 = (2 * local + rank) * QBN;
  } else {
    const int pm = local / nt;
    tl.mc = true;
    mi = 2 * pm + rank;
    tl.n0 = (local - pm * nt) * QBN;
  }
  tl.nh = max(0, min(2, (g.N - tl.n0) / QHN));
  tl.ghost = mi >= mt || tl.nh == 0;
  if constexpr (KIND == MxKind::kWgrad) {
    tl.m0 = mi * QBM;
    tl.k0 = s_off[lo];
    const int kr = s_off[lo + 1] - s_off[lo];
    tl.kblocks = (kr + QBK - 1) / QBK;
    tl.klast = kr - (tl.kblocks - 1) * QBK;
    tl.row0 = 0;
    tl.rows = 0;
  } else {
    tl.row0 = s_off[lo] + mi * QBM;
    tl.rows = tl.ghost ? 0 : min(QBM, s_off[lo + 1] - tl.row0);
    tl.kblocks = g.K / QBK;
    tl.klast = QBK;
    tl.m0 = 0;
    tl.k0 = 0;
  }
  return tl;
}

// 32 fp32 accumulator columns -> 32 bf16 at p (64 bytes)
__device__ __forceinline__ void mx_store_row32(uint16_t* p, const uint32_t (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(p + 8 * k) = make_uint4(
        pack_bf16x2(__uint_as_float(v[8 * k + 0]), __uint_as_float(v[8 * k + 1])),
        pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
        pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
        pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
}

// GroupGemm + Quantize ([TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩"):
// 32 fp32 accumulator columns of one row -> 32 bf16 at p, and the row-wise
// MXFP8 block of those bf16 values: 32 codes at q, the E8M0 scale at *s
__device__ __forceinline__ void mx_store_quant_row32(uint16_t* p, uint8_t* q, uint8_t* s,
                                                     const uint32_t (&v)[32]) {
  uint32_t pk[16];
  float f[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    f[2 * i] = bf16_lo(pk[i]);
    f[2 * i + 1] = bf16_hi(pk[i]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(p + 8 * k) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
  uint32_t qw[8];
  *s = static_cast<uint8_t>(mx_quant32(f, qw));
  uint4* pq = reinterpret_cast<uint4*>(q);
  pq[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  pq[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
}

// dA columns col..col+31 of one row -> dH (same interleaving as H)
template <int ACT>
__device__ __forceinline__ void mx_dact_row32(const MxGemmArgs& g, long long grow, int col,
                                              const uint32_t (&r)[32]) {
  if constexpr (ACT == MOE_ACT_SRELU) {
    const uint16_t* hp = g.aux + grow * g.ld_aux + col;
    uint16_t* p = g.out + grow * g.ldo + col;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = pack_bf16x2(2.f * fmaxf(bf16_lo(hw[i]), 0.f) * __uint_as_float(r[8 * v + 2 * i]),
                           2.f * fmaxf(bf16_hi(hw[i]), 0.f) * __uint_as_float(r[8 * v + 2 * i + 1]));
      *reinterpret_cast<uint4*>(p + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    const uint16_t* hp = g.aux + grow * g.ld_aux + 2 * col;
    uint16_t* p = g.out + grow * g.ldo + 2 * col;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};  // (gate, up) pairs
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float gg = bf16_lo(hw[i]), uu = bf16_hi(hw[i]);
        const float da = __uint_as_float(r[4 * v + i]);
        float ph, dph;
        gate_phi_dphi<ACT>(gg, ph, dph);
        o[i] = pack_bf16x2(da * uu * dph, da * ph);
      }
      *reinterpret_cast<uint4*>(p + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Persistent warp-specialised block-scaled grouped GEMM in 2-CTA clusters:
// warp 0 TMA producer (operand tiles by tensor maps, B halves multicast
// within the pair, scale chunks by bulk copies), warp 1 TMEM owner and MMA
// issuer (tcgen05.mma ... block_scale; the scale chunks of a stage go to TMEM
// with tcgen05.cp; its commit frees the stage in both CTAs), warps 2-9
// epilogue in two warpgroups, one per 128-column half of the tile.
template <MxKind KIND, int ACT, bool QOUT>
__global__ void __launch_bounds__(QTHREADS, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const MxGemmArgs g) {
  constexpr bool W = (KIND == MxKind::kWgrad);
  constexpr bool B_MN = (KIND == MxKind::kFc2);
  constexpr uint32_t IDESC = idesc_mx(QBM, QHN, false, B_MN);
  constexpr int NST = QCfg<KIND>::stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* staging = smem + NST * QSTAGE_BYTES;               // one box per epilogue warp
  uint8_t* zero_box = staging + QEPI_WARPS * QBOX_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + QCfg<KIND>::stg_bytes);
  uint64_t* empty_bar = full_bar + NST;
  uint64_t* tfull_bar = empty_bar + NST;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* drain_bar = tempty_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_ts = s_off + (g.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int unit0 = blockIdx.x / QCL;     // this cluster's first work unit
  const int unit_step = gridDim.x / QCL;  // clusters in the grid

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], QCL);  // one commit from each CTA's MMA warp
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, QEPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (W) prefetch_tmap(&tmC);
  }
  if (W && warp >= 2) {  // epilogue threads clear the zero box
    for (int i = threadIdx.x - 64; i < QBOX_BYTES / 16; i += 32 * QEPI_WARPS)
      reinterpret_cast<uint4*>(zero_box)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, QTMEM_COLS);
  if (warp == 2) {
    // offsets: non-decreasing multiples of 32 within [0, M_cap]
    bool bad = false;
    for (int i = lane; i <= g.E; i += 32) {
      const int v = g.offsets[i];
      if (v < 0 || v > g.M_cap || (v & 31)) bad = true;
      s_off[i] = min(max(v, 0), g.M_cap) & ~31;
    }
    __syncwarp();
    if (lane == 0) {
      int prev = 0;
      for (int i = 0; i <= g.E; ++i) {
        if (s_off[i] < prev) { bad = true; s_off[i] = prev; }
        prev = s_off[i];
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) set_err(g.err, MOE_DEV_BAD_OFFSETS);
    __syncwarp();
    int carry = 0;
    for (int base = 0; base < g.E; base += 32) {
      const int e = base + lane;
      const int t = (e < g.E) ? mx_tiles_of_expert<KIND>(g, s_off, e) : 0;
      int v = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (e < g.E) s_ts[e] = carry + v - t;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_ts[g.E] = carry;
  }
  tc_fence_before();
  cluster_sync();  // the peer's barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_ts[g.E];

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool issued[NST];
      uint32_t ipar[NST];
      for (int i = 0; i < NST; ++i) { issued[i] = false; ipar[i] = 0; }
      bool ok = true;
      const long long kc_n = g.K / QBK, nq = g.N / QHN, rq = g.R / QBM;
      for (int t = unit0; t < total && ok; t += unit_step) {
        const QTile tl = mx_decode<KIND>(g, s_off, s_ts, t, rank);
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * QSTAGE_BYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sa + QSF_OFF;
          uint64_t* fb = &full_bar[stage];
          // B's halves land in this stage whoever fetched them; A and the
          // scale chunks (small, loaded by each CTA itself) only for a real tile
          mbar_arrive_expect_tx(fb, tl.nh * QBH_BYTES + (tl.ghost ? 0 : QA_BYTES + 512 + tl.nh * 512));
          long long ca, cb0, cstep;  // scale chunks: A, B half 0, B half 1 - half 0
          if constexpr (W) {
            const int kc = tl.k0 + kb * QBK;
            if (!tl.ghost) tma_load_2d(sa, &tmA, fb, kc, tl.m0);
            for (int h = 0; h < tl.nh; ++h) {
              if (tl.mc && h != rank) continue;
              if (tl.mc) tma_load_2d_mc(sb + h * QBH_BYTES, &tmB, fb, kc, tl.n0 + h * QHN, kQPair);
              else tma_load_2d(sb + h * QBH_BYTES, &tmB, fb, kc, tl.n0 + h * QHN);
            }
            ca = static_cast<long long>(kc / 32) * rq + tl.m0 / QBM;
            cb0 = static_cast<long long>(kc / 32) * nq + tl.n0 / QHN;
            cstep = 1;
          } else {
            if (!tl.ghost) tma_load_2d(sa, &tmA, fb, kb * QBK, tl.row0);
            ca = static_cast<long long>(tl.row0 / 32) * kc_n + kb;
            if constexpr (B_MN) {
              for (int h = 0; h < tl.nh; ++h) {
                if (tl.mc && h != rank) continue;
                if (tl.mc)
                  tma_load_3d_mc(sb + h * QBH_BYTES, &tmB, fb, tl.n0 + h * QHN, kb * QBK, tl.e, kQPair);
                else tma_load_3d(sb + h * QBH_BYTES, &tmB, fb, tl.n0 + h * QHN, kb * QBK, tl.e);
              }
              cb0 = (static_cast<long long>(tl.e) * kc_n + kb) * nq + tl.n0 / QHN;
              cstep = 1;
            } else {
              for (int h = 0; h < tl.nh; ++h) {
                if (tl.mc && h != rank) continue;
                const int rb = tl.e * g.N + tl.n0 + h * QHN;
                if (tl.mc) tma_load_2d_mc(sb + h * QBH_BYTES, &tmB, fb, kb * QBK, rb, kQPair);
                else tma_load_2d(sb + h * QBH_BYTES, &tmB, fb, kb * QBK, rb);
              }
              cb0 = ((static_cast<long long>(tl.e) * g.N + tl.n0) / QHN) * kc_n + kb;
              cstep = kc_n;
            }
          }
          if (!tl.ghost) {
            bulk_load(ssf, g.a_s + ca * 512, 512, fb);
            for (int h = 0; h < tl.nh; ++h)
              bulk_load(ssf + 512 * (1 + h), g.b_s + (cb0 + h * cstep) * 512, 512, fb);
          }
          issued[stage] = true;
          ipar[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        for (int i = 0; i < NST; ++i)
          if (issued[i]) {
            const uint32_t a = smem_u32(&full_bar[i]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(a, ipar[i]) && globaltimer_ns() - t0 < kWaitLimitNs) {}
          }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int t = unit0; t < total && ok; t += unit_step, ++local) {
      const QTile tl = mx_decode<KIND>(g, s_off, s_ts, t, rank);
      // the accumulator is free once the epilogue has read the previous tile
      if (lane == 0) ok = mbar_wait(tempty_bar, (local & 1) ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      for (int kb = 0; kb < tl.kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&full_bar[stage], phase, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0 && !tl.ghost) {
          uint8_t* sa = smem + stage * QSTAGE_BYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sa + QSF_OFF;
          const uint32_t sf_t = tmem_base + QSF_TMEM + stage * QSF_COLS;
          tmem_cp_sf(sf_t, sdesc_sf(smem_u32(ssf)));
          for (int h = 0; h < tl.nh; ++h)
            tmem_cp_sf(sf_t + 4 * (1 + h), sdesc_sf(smem_u32(ssf + 512 * (1 + h))));
          const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
          // an expert's last reduction step of a weight gradient holds
          // klast (a multiple of 32) of its rows: one MMA per 32 of them
          const int kk_n = (W && kb == tl.kblocks - 1) ? tl.klast / 32 : QBK / 32;
          for (int kk = 0; kk < kk_n; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint32_t id = IDESC | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
            for (int h = 0; h < tl.nh; ++h) {
              const uint32_t bh = b0 + h * QBH_BYTES;
              const uint64_t bd = B_MN ? sdesc_sw128(bh + kk * 4096, QBH_BYTES, 1024)
                                       : sdesc_sw128(bh + kk * 32, 16, 1024);
              umma_mx(tmem_base + h * QHN, ad, bd, id, sf_t, sf_t + 4 * (1 + h),
                      (kb > 0 || kk > 0) ? 1u : 0u);
            }
          }
        }
        // the stage is free in both CTAs once both MMA warps have read it
        if (lane == 0) umma_commit_mc(&empty_bar[stage], kQPair);
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(tfull_bar);
      __syncwarp();
    }
    if (!ok && lane == 0) {
      umma_commit(drain_bar);
      const uint32_t a = smem_u32(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quadrant
    const int wg = (warp - 2) >> 2;      // 128-column half of the tile
    const int r = q * 32 + lane;
    uint8_t* my_box = staging + (warp - 2) * QBOX_BYTES;
    int local = 0;
    for (int t = unit0; t < total; t += unit_step, ++local) {
      const QTile tl = mx_decode<KIND>(g, s_off, s_ts, t, rank);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(tfull_bar, local & 1, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const bool zero = W && tl.kblocks == 0;
      // accumulating weight gradients leave an empty expert's untouched
      const bool mine = wg < tl.nh && !tl.ghost && !(zero && g.accumulate);
      uint32_t v[4][32];
      if (mine && !zero) {
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + wg * QHN;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tb + c * 32, v[c]);
        tmem_wait_ld();
      }
      // release the accumulator: the next tile's MMAs may start
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar);
      if (!mine) continue;
      const int col0 = tl.n0 + wg * QHN;
      if constexpr (W) {
        if (g.accumulate && !zero) {
          const uint16_t* op = g.out + (static_cast<long long>(tl.e) * g.R + tl.m0 + q * 32 + lane) * g.N + col0;
#pragma unroll
          for (int c = 0; c < 4; ++c) add_bf16_row32(op + 32 * c, v[c]);
        }
        if (zero) {
          // expert with no rows: its weight gradient is zero
          if (lane == 0) {
            tma_store_3d(&tmC, zero_box, col0, tl.m0 + q * 32, tl.e);
            tma_store_3d(&tmC, zero_box, col0 + 64, tl.m0 + q * 32, tl.e);
            bulk_commit();
          }
          __syncwarp();
        } else {
          // stage each 32-row x 64-column box (128-byte swizzle: 16-byte
          // chunk j of row r at j ^ (r % 8)) and write it with a TMA store
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (lane == 0) bulk_wait_read_0();     // the box's previous store has read it
            __syncwarp();
            uint8_t* row = my_box + lane * 128;
            const int sw = lane & 7;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t (&src)[32] = v[2 * h + (j >> 2)];
              const int b = 8 * (j & 3);
              *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) = make_uint4(
                  pack_bf16x2(__uint_as_float(src[b + 0]), __uint_as_float(src[b + 1])),
                  pack_bf16x2(__uint_as_float(src[b + 2]), __uint_as_float(src[b + 3])),
                  pack_bf16x2(__uint_as_float(src[b + 4]), __uint_as_float(src[b + 5])),
                  pack_bf16x2(__uint_as_float(src[b + 6]), __uint_as_float(src[b + 7])));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, my_box, col0 + h * 64, tl.m0 + q * 32, tl.e);
              bulk_commit();
            }
          }
        }
      } else {
        if (r < tl.rows) {
          const long long grow = tl.row0 + r;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if constexpr (KIND == MxKind::kDgradAct) mx_dact_row32<ACT>(g, grow, col0 + c * 32, v[c]);
            else if (QOUT)
              mx_store_quant_row32(g.out + grow * g.ldo + col0 + c * 32,
                                   g.q_out + grow * g.N + col0 + c * 32,
                                   g.s_out + grow * (g.N / 32) + (col0 + c * 32) / 32, v[c]);
            else mx_store_row32(g.out + grow * g.ldo + col0 + c * 32, v[c]);
          }
        }
      }
    }
    if (W && lane == 0) bulk_wait_all();  // staged stores done before the CTA exits
    __syncwarp();
  }
  tc_fence_before();
  // no CTA leaves while its peer may still multicast into it or arrive on it
  cluster_sync();
  if (*abort_flag && threadIdx.x == 0) set_err(g.err, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, QTMEM_COLS);
  }
}

template <MxKind KIND, int ACT, bool QOUT = false>
cudaError_t launch_mx_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const MxGemmArgs& g, int num_sms, cudaStream_t st) {
  auto kern = mx_gemm_kernel<KIND, ACT, QOUT>;
  const size_t smem = mx_smem_bytes<KIND>(MOE_MAX_EXPERTS);
  // grid size and shared-memory attribute, set up once per device and
  // instantiation
  static int grid_of[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = QCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(QTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int& grid = grid_of[dev];
  if (grid == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    const int most = num_sms / QCL;
    grid = QCL * ((clusters > 0 && clusters < most) ? clusters : most);
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, g);
}

}  // namespace

cudaError_t launch_mx_quantize_weights(const uint16_t* w2, int E, int n, int d,
                                       const int32_t* offsets, uint8_t* q, uint8_t* s,
                                       uint8_t* q_rows, uint8_t* s_rows, int num_sms,
                                       cudaStream_t st) {
  if (q_rows) {
    const long long threads = static_cast<long long>(E) * (n / 32) * (d / 128) * 32;
    const long long want = (threads + 255) / 256;
    const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
    mx_quantize_w2_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
        reinterpret_cast<const uint4*>(w2), E, n, d, offsets, reinterpret_cast<uint2*>(q), s,
        reinterpret_cast<uint2*>(q_rows), s_rows);
  } else {
    // the forward alone: the one-direction kernel streams faster (measured
    // on the 256-expert W2: 1.64 ms against 1.86 ms for the two-direction
    // kernel's column half)
    const long long threads = static_cast<long long>(E) * (n / 32) * (d / 8);
    const long long want = (threads + 255) / 256;
    const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
    mx_quantize_weights_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
        reinterpret_cast<const uint4*>(w2), E, n, d, offsets, reinterpret_cast<uint2*>(q), s);
  }
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_act(const uint16_t* src, int rows, int cols, const int32_t* offsets,
                                   int E, uint8_t* q, uint8_t* s, uint8_t* qT, uint8_t* sT,
                                   int32_t* err, bool tiled, int num_sms, cudaStream_t st) {
  if (tiled) {
    if (cols % 128) return cudaErrorInvalidValue;   // the tiles cover 128-column groups
    // as many blocks as the SMs hold at once: each loads the offsets once
    static int per_sm = 0;
    if (per_sm <= 0) {
      int nb = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, mx_quantize_act_w_kernel, 256, 0) !=
              cudaSuccess || nb <= 0)
        nb = 1;
      per_sm = nb;
    }
    const long long warps = static_cast<long long>(rows / 32) * (cols / 128);
    const long long want = (warps * 32 + 255) / 256;
    const long long cap = static_cast<long long>(per_sm) * num_sms;
    const int blocks = static_cast<int>(want < cap ? want : cap);
    mx_quantize_act_w_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
        reinterpret_cast<const uint4*>(src), rows, cols, offsets, E, reinterpret_cast<uint2*>(q), s,
        qT, sT, err);
    return cudaGetLastError();
  }
  const long long warps = static_cast<long long>(rows / 32) * (cols / 32);
  const long long want = (warps * 32 + 255) / 256;
  const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
  mx_quantize_act_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(src), rows, cols, offsets, E, q, s, qT, sT, err);
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_rows_w(const uint16_t* src, long long rows, int cols,
                                      const int32_t* offsets, long long rows_per_e, uint8_t* q,
                                      uint8_t* s, int num_sms, cudaStream_t st) {
  // one warp per 32 blocks (rows * cols / 32 is a multiple of 32: rows and
  // cols are multiples of 128)
  const long long threads = rows * (cols / 32);
  const long long want = (threads + 255) / 256;
  const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
  mx_quantize_rows_w_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(src), rows, cols, offsets, rows_per_e,
      reinterpret_cast<uint2*>(q), s);
  return cudaGetLastError();
}

cudaError_t launch_mx_retile_t(const uint8_t* sT, int rows, int cols, const int32_t* offsets,
                               int E, uint8_t* out, int num_sms, cudaStream_t st) {
  const long long threads = static_cast<long long>(cols) * (rows / 32);
  const long long want = (threads + 255) / 256;
  const int blocks = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
  mx_retile_t_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(sT, rows, cols, offsets, E, out);
  return cudaGetLastError();
}

cudaError_t launch_mx_gemm(MxKind kind, int act, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const MxGemmArgs& g, int num_sms,
                           cudaStream_t st) {
  switch (kind) {
    // the quantising epilogue (GroupGemm + Quantize) is its own instantiation,
    // so that the plain one keeps its registers
    case MxKind::kFc2:
      return g.q_out ? launch_mx_t<MxKind::kFc2, 0, true>(ta, tb, tc, g, num_sms, st)
                     : launch_mx_t<MxKind::kFc2, 0>(ta, tb, tc, g, num_sms, st);
    case MxKind::kDgrad:
      return g.q_out ? launch_mx_t<MxKind::kDgrad, 0, true>(ta, tb, tc, g, num_sms, st)
                     : launch_mx_t<MxKind::kDgrad, 0>(ta, tb, tc, g, num_sms, st);
    case MxKind::kWgrad: return launch_mx_t<MxKind::kWgrad, 0>(ta, tb, tc, g, num_sms, st);
    case MxKind::kDgradAct:
      switch (act) {
        case MOE_ACT_SWIGLU: return launch_mx_t<MxKind::kDgradAct, MOE_ACT_SWIGLU>(ta, tb, tc, g, num_sms, st);
        case MOE_ACT_GEGLU: return launch_mx_t<MxKind::kDgradAct, MOE_ACT_GEGLU>(ta, tb, tc, g, num_sms, st);
        case MOE_ACT_SRELU: return launch_mx_t<MxKind::kDgradAct, MOE_ACT_SRELU>(ta, tb, tc, g, num_sms, st);
        default: return cudaErrorInvalidValue;
      }
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
