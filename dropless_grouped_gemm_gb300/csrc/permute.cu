// permute.cu - expert-major gather (permute) and weighted combine
// (unpermute) with the optional router-score gradient.
//
// [TE] "최적화 2: NCCL EP": dispatch permutes token rows into the experts'
// order, combine returns them and accumulates each token's expert outputs.
// [Sonic] "역전파 계산 그래프 재작성하기": dS_{t,e} = <dO_t, Y_{e,t}>.
//
// All three are HBM-bound: 16-byte vector loads and stores, grid-stride
// over work items with as many CTAs as the SMs hold at once.  A work item is
// a row (permute), a 2 KB segment of one token's row (combine) or one
// (token, slot) pair (router gradient): a 7,168-wide layer of 4,096 tokens
// then gives the combine and the router gradient tens of thousands of
// items instead of one per token.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 32;

__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float s) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(s * bf16_lo(w[i]), s * bf16_hi(w[i]));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// 16-byte vectors per combine work item: 2 KB of a row
constexpr int kSeg = 128;
// slots of one token loaded together by the combine
constexpr int kSlots = 8;

// dst[r] = (scale ? scale[p] : 1) * src[p / k], p = pair_of_row[r]; 0 if p is
// outside [0, P).  Work item: a whole row.  (2 KB segments, as the combine
// takes them, measured 3.5% slower here: the pass is bound by its writes.)
__global__ void __launch_bounds__(kThreads)
    permute_kernel(const uint4* __restrict__ src, const float* __restrict__ scale,
                   const int32_t* __restrict__ pair_of_row, int P, int k, int dv, int M_cap,
                   uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); r < M_cap;
       r += gridDim.x * kRowsPerBlock) {
    const int p = pair_of_row[r];
    uint4* out = dst + static_cast<long long>(r) * dv;
    // streaming (evict-first) stores: the permuted copy is far larger than
    // L2 and is read back by the next GEMM from DRAM anyway (measured 6%
    // faster than plain stores on the Zipf layer)
    if (p < 0 || p >= P) {
      for (int v = lane; v < dv; v += 32) __stcs(out + v, make_uint4(0, 0, 0, 0));
      continue;
    }
    const uint4* in = src + static_cast<long long>(p / k) * dv;
    if (scale == nullptr) {
      int v = lane;
      for (; v + 96 < dv; v += 128) {
        const uint4 a = __ldg(in + v), b = __ldg(in + v + 32), c = __ldg(in + v + 64),
                    d = __ldg(in + v + 96);
        __stcs(out + v, a); __stcs(out + v + 32, b); __stcs(out + v + 64, c); __stcs(out + v + 96, d);
      }
      for (; v < dv; v += 32) __stcs(out + v, __ldg(in + v));
    } else {
      const float s = scale[p];
      for (int v = lane; v < dv; v += 32) __stcs(out + v, scale_bf16x8(__ldg(in + v), s));
    }
  }
}

// The same permuted copy in token order, from both maps: a warp reads a
// 2 KB segment of a token's row once and writes it to each of the token's k
// rows (row_of_pair), scaled per pair when scale is given; a pair whose row
// lies outside [0, M_cap), or is not mapped back to it by pair_of_row, writes
// nothing.  The row-order kernel above reads each token row once per pair
// from whichever SM takes the destination row, and on the two-die GB300 most
// of those reads miss the reading die's L2 (3.7x the token tensor from DRAM
// on the Zipf layer).  The token work items are 2 KB segments of a row; the
// items after them are the M_cap rows, one each: a row that no valid pair
// maps to (pair_of_row outside [0, P)) is zeroed.  (Groups of 32 rows put a
// run of pad rows on one warp: 151 against 137 us for the row-order kernel
// on a layer with 7,936 pad rows.)
__global__ void __launch_bounds__(kThreads)
    permute_tokens_kernel(const uint4* __restrict__ src, const float* __restrict__ scale,
                          const int32_t* __restrict__ row_of_pair,
                          const int32_t* __restrict__ pair_of_row, int T, int k, int dv,
                          int M_cap, uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const long long P = static_cast<long long>(T) * k;
  const int nseg = (dv + kSeg - 1) / kSeg;
  const long long tok_items = static_cast<long long>(T) * nseg;
  const long long items = tok_items + M_cap;
  for (long long it = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
       it < items; it += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    if (it < tok_items) {
      const int t = static_cast<int>(it / nseg);
      const uint4* in = src + static_cast<long long>(t) * dv;
      {
        const int v0 = static_cast<int>(it - static_cast<long long>(t) * nseg) * kSeg;
        uint4 x[kSeg / 32];
#pragma unroll
        for (int i = 0; i < kSeg / 32; ++i) {
          const int v = v0 + lane + 32 * i;
          x[i] = (v < dv) ? __ldg(in + v) : make_uint4(0, 0, 0, 0);
        }
        for (int j = 0; j < k; ++j) {
          const long long p = static_cast<long long>(t) * k + j;
          const int r = row_of_pair[p];
          if (r < 0 || r >= M_cap || pair_of_row[r] != p) continue;
          uint4* out = dst + static_cast<long long>(r) * dv;
          const float sc = scale ? scale[p] : 1.0f;
#pragma unroll
          for (int i = 0; i < kSeg / 32; ++i) {
            const int v = v0 + lane + 32 * i;
            if (v < dv) __stcs(out + v, scale ? scale_bf16x8(x[i], sc) : x[i]);
          }
        }
      }
    } else {
      const int r = static_cast<int>(it - tok_items);
      const int p = pair_of_row[r];
      if (p < 0 || p >= P) {
        uint4* out = dst + static_cast<long long>(r) * dv;
        for (int v = lane; v < dv; v += 32) __stcs(out + v, make_uint4(0, 0, 0, 0));
      }
    }
  }
}

// dst[t] = sum_j w_tj src[row(t,j)] (fp32, j ascending).  Work item:
// segment sg of token t; the rows of up to kSlots slots are loaded together
// before they are added in slot order, so their latencies overlap.
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const uint4* __restrict__ src, const float* __restrict__ probs,
                   const int32_t* __restrict__ row_of_pair, int T, int k, int dv, int M_cap,
                   uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int nseg = (dv + kSeg - 1) / kSeg;
  const long long items = static_cast<long long>(T) * nseg;
  for (long long it = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
       it < items; it += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const int t = static_cast<int>(it / nseg);
    const int v0 = static_cast<int>(it - static_cast<long long>(t) * nseg) * kSeg;
    const int v1 = min(v0 + kSeg, dv);
    const long long pair0 = static_cast<long long>(t) * k;
    uint4* out = dst + static_cast<long long>(t) * dv;
    for (int v = v0 + lane; v < v1; v += 32) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int j0 = 0; j0 < k; j0 += kSlots) {
        uint4 y[kSlots];
        float w[kSlots];
        bool ok[kSlots];
#pragma unroll
        for (int jj = 0; jj < kSlots; ++jj) {
          const int j = j0 + jj;
          const int row = (j < k) ? row_of_pair[pair0 + j] : -1;
          ok[jj] = row >= 0 && row < M_cap;
          w[jj] = (ok[jj] && probs) ? probs[pair0 + j] : 1.0f;
          y[jj] = ok[jj] ? __ldg(src + static_cast<long long>(row) * dv + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int jj = 0; jj < kSlots; ++jj) {
          if (!ok[jj]) continue;
          const uint32_t yw[4] = {y[jj].x, y[jj].y, y[jj].z, y[jj].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(w[jj], bf16_lo(yw[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(w[jj], bf16_hi(yw[i]), acc[2 * i + 1]);
          }
        }
      }
      out[v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// dprobs[t*k+j] = <dO[t], src[row(t,j)]> (fp32; per lane in increasing
// vector order, then a fixed butterfly across lanes: deterministic).  Work
// item: one pair; four vectors of both rows are loaded before they are
// accumulated in order.
__global__ void __launch_bounds__(kThreads)
    router_grad_kernel(const uint4* __restrict__ src, const uint4* __restrict__ dO,
                       const int32_t* __restrict__ row_of_pair, int T, int k, int dv, int M_cap,
                       float* __restrict__ dprobs) {
  const int lane = threadIdx.x & 31;
  const long long P = static_cast<long long>(T) * k;
  for (long long p = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
       p < P; p += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const int row = row_of_pair[p];
    float acc = 0.f;
    if (row >= 0 && row < M_cap) {
      const uint4* g = dO + (p / k) * dv;
      const uint4* y = src + static_cast<long long>(row) * dv;
      auto dot8 = [&](uint4 a, uint4 b) {
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(bf16_lo(aw[i]), bf16_lo(bw[i]), acc);
          acc = fmaf(bf16_hi(aw[i]), bf16_hi(bw[i]), acc);
        }
      };
      int v = lane;
      for (; v + 96 < dv; v += 128) {
        const uint4 a0 = __ldg(g + v), a1 = __ldg(g + v + 32), a2 = __ldg(g + v + 64),
                    a3 = __ldg(g + v + 96);
        const uint4 b0 = __ldg(y + v), b1 = __ldg(y + v + 32), b2 = __ldg(y + v + 64),
                    b3 = __ldg(y + v + 96);
        dot8(a0, b0); dot8(a1, b1); dot8(a2, b2); dot8(a3, b3);
      }
      for (; v < dv; v += 32) dot8(__ldg(g + v), __ldg(y + v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) dprobs[p] = acc;
  }
}

// dprobs[p] = sum of the row's partial <dA', A> (routed backward), summed in
// a fixed order; 0 for pairs without a row
__global__ void __launch_bounds__(kThreads)
    router_grad_rows_kernel(const float* __restrict__ ds_part, int n_parts,
                            const int32_t* __restrict__ row_of_pair, int P, int M_cap,
                            float* __restrict__ dprobs) {
  for (int p = blockIdx.x * kThreads + threadIdx.x; p < P; p += gridDim.x * kThreads) {
    const int row = row_of_pair[p];
    float s = 0.f;
    if (row >= 0 && row < M_cap) {
      const float* q = ds_part + static_cast<long long>(row) * n_parts;
      for (int i = 0; i < n_parts; ++i) s += q[i];
    }
    dprobs[p] = s;
  }
}

// Grid of a grid-stride pass over `items` warp work items: no more blocks
// than the SMs hold at once (the occupancy the runtime reports for this
// kernel, looked up once into *per_sm), so that no block waits for a second
// wave while the others stream.
int grid_for(const void* kernel, int* per_sm, long long items, int num_sms) {
  if (*per_sm <= 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess ||
        n <= 0)
      n = 1;
    *per_sm = n;
  }
  const long long want = (items + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long cap = static_cast<long long>(*per_sm) * num_sms;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

int g_permute_per_sm = 0, g_permute_tokens_per_sm = 0, g_combine_per_sm = 0,
    g_router_grad_per_sm = 0;

}  // namespace

cudaError_t launch_permute(const uint16_t* src, const float* scale, const int32_t* pair_of_row,
                           int T, int k, int d, int M_cap, uint16_t* dst, int num_sms,
                           cudaStream_t s) {
  if (M_cap <= 0) return cudaSuccess;
  permute_kernel<<<grid_for(reinterpret_cast<const void*>(permute_kernel), &g_permute_per_sm,
                            M_cap, num_sms),
                   kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(src), scale, pair_of_row, T * k, k, d / 8, M_cap,
      reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_permute_tokens(const uint16_t* src, const float* scale,
                                  const int32_t* row_of_pair, const int32_t* pair_of_row, int T,
                                  int k, int d, int M_cap, uint16_t* dst, int num_sms,
                                  cudaStream_t s) {
  if (M_cap <= 0) return cudaSuccess;
  const long long items = static_cast<long long>(T) * ((d / 8 + kSeg - 1) / kSeg) + M_cap;
  permute_tokens_kernel<<<grid_for(reinterpret_cast<const void*>(permute_tokens_kernel),
                                   &g_permute_tokens_per_sm, items, num_sms),
                          kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(src), scale, row_of_pair, pair_of_row, T, k, d / 8, M_cap,
      reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const uint16_t* src, const float* probs,
                             const int32_t* row_of_pair, int T, int k, int d, int M_cap,
                             uint16_t* dst,
                             const uint16_t* dO, float* dprobs, int num_sms, cudaStream_t s,
                             int* launches) {
  *launches = 0;
  if (T <= 0) return cudaSuccess;
  const long long nseg = (d / 8 + kSeg - 1) / kSeg;
  if (dst) {
    combine_kernel<<<grid_for(reinterpret_cast<const void*>(combine_kernel), &g_combine_per_sm,
                                      T * nseg, num_sms),
                     kThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(src), probs, row_of_pair, T, k, d / 8, M_cap,
        reinterpret_cast<uint4*>(dst));
    ++*launches;
  }
  if (dprobs) {
    router_grad_kernel<<<grid_for(reinterpret_cast<const void*>(router_grad_kernel),
                                  &g_router_grad_per_sm, static_cast<long long>(T) * k, num_sms),
                         kThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<const uint4*>(dO), row_of_pair,
        T, k, d / 8, M_cap, dprobs);
    ++*launches;
  }
  return cudaGetLastError();
}

cudaError_t launch_router_grad_rows(const float* ds_part, int n_parts, const int32_t* row_of_pair,
                                   int P, int M_cap, float* dprobs, int num_sms, cudaStream_t s) {
  if (P <= 0) return cudaSuccess;
  const long long want = (P + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(want < 4LL * num_sms ? want : 4LL * num_sms);
  router_grad_rows_kernel<<<grid, kThreads, 0, s>>>(ds_part, n_parts, row_of_pair, P, M_cap,
                                                    dprobs);
  return cudaGetLastError();
}

}  // namespace moe
