// mx_quant.cu - MXFP8 quantisers (OCP MX v1.0: E4M3 codes, E8M0 scale per
// 32 values; block rule in mx.cuh):
//   * mx_quantize_weights / mx_quantize_w2: W2 [E, n, d] with blocks of 32
//     rows (FC2's reduction index) per column, and from the same read the
//     copy with blocks along d (FC2-dgrad's), scales in the MMA tiles.
//   * mx_quantize_rows_w: any weight viewed as [rows, K] with blocks along
//     K (the reduction index of a data gradient), scales in weight tiles.
//   * mx_quantize_act_w / mx_quantize_act: group-aware quantisers of a
//     ragged [rows, cols] activation: row-wise 1x32 blocks, plus the
//     transposed copy with column-wise 32x1 blocks that never cross an
//     expert's rows; scales in the tiles the GEMM reads, or plain.
//   * mx_retile_t: plain transposed scales -> the weight gradient's K tiles.
// With the routing offsets the weight quantisers skip experts without rows.
// [CuTe] "무엇을 해결하려는가" and "핵심 아이디어": MXFP8 output and transposed
// output; [TE] "Transformer Engine이 제공하는 세 가지 구성 요소": group-aware
// MXFP8 quantisation.
#include <cuda_runtime.h>

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
  // 32-bit warp indices (the launch checks E * n * d < 2^40): two 32-bit
  // divisions per iteration split one into expert, row block and column chunk
  const uint32_t cw = static_cast<uint32_t>(d / 128);      // warps per 32-row block
  const uint32_t nb = static_cast<uint32_t>(n / 32);       // row blocks of one expert
  const uint32_t nwarps = static_cast<uint32_t>(ne) * nb * cw;
  for (uint32_t wi = (blockIdx.x * blockDim.x + threadIdx.x) / 32; wi < nwarps;
       wi += gridDim.x * blockDim.x / 32) {
    const uint32_t eb = wi / cw;
    const int c8 = static_cast<int>(wi - eb * cw) * 16 + (lane & 15);
    const uint32_t eu = eb / nb;
    const int b = static_cast<int>(eb - eu * nb);
    const int e = offsets ? s_list[eu] : static_cast<int>(eu);
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
  const uint32_t cb_n = static_cast<uint32_t>(cols / 32);
  const int ne = used_experts(offsets, static_cast<int>(rows / rows_per_e), s_list, &s_count);
  // warp and block indices inside the used experts fit in 32 bits (the
  // launch checks rows * cols < 2^37): one 32-bit division per iteration
  // finds the expert, one more the row of the warp's first block
  const uint32_t warps_e = static_cast<uint32_t>(rows_per_e * cb_n / 32);
  const uint32_t nwarps = static_cast<uint32_t>(ne) * warps_e;
  const long long tiles_e = rows_per_e / 128;        // 128-row scale tiles of one expert
  for (uint32_t wi = (blockIdx.x * blockDim.x + threadIdx.x) / 32; wi < nwarps;
       wi += gridDim.x * blockDim.x / 32) {
    const uint32_t eu = wi / warps_e;
    const uint32_t local = wi - eu * warps_e;
    const long long e = offsets ? s_list[eu] : eu;
    const long long g0 = (e * warps_e + local) * 32;  // first block of the warp
    uint32_t x[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(src + g0 * 4 + 32 * k + lane);
      x[k][0] = v.x; x[k][1] = v.y; x[k][2] = v.z; x[k][3] = v.w;
    }
    // row (inside the expert) and column block of the warp's first block
    const uint32_t b0 = local * 32;
    const uint32_t rl0 = b0 / cb_n;
    const uint32_t cb0 = b0 - rl0 * cb_n;
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
        // this block: b0 + 8k + lane/4, at most 31 blocks past the first
        uint32_t cb = cb0 + 8 * k + (lane >> 2);
        uint32_t rl = rl0;
        while (cb >= cb_n) { cb -= cb_n; ++rl; }
        const long long chunk = (e * tiles_e + (rl >> 7)) * (cols / 128) + cb / 4;
        s[chunk * 512 + mx_chunk_off(static_cast<int>(rl & 127), cb & 3)] = static_cast<uint8_t>(sc);
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

}  // namespace

cudaError_t launch_mx_quantize_weights(const uint16_t* w2, int E, int n, int d,
                                       const int32_t* offsets, uint8_t* q, uint8_t* s,
                                       uint8_t* q_rows, uint8_t* s_rows, int num_sms,
                                       cudaStream_t st) {
  if (q_rows) {
    if (static_cast<long long>(E) * n * d >= (1LL << 40)) return cudaErrorInvalidValue;
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
  if (rows * cols >= (1LL << 37)) return cudaErrorInvalidValue;   // 32-bit indices in the kernel
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

}  // namespace moe
