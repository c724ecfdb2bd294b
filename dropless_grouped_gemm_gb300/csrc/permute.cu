// permute.cu - expert-major gather (permute) and weighted combine
// (unpermute) with the optional router-score gradient.
//
// [TE] "최적화 2: NCCL EP": dispatch permutes token rows into the experts'
// order, combine returns them and accumulates each token's expert outputs.
// [Sonic] "역전파 계산 그래프 재작성하기": dS_{t,e} = <dO_t, Y_{e,t}>.
//
// Both kernels are HBM-bound row copies: one warp per row, 16-byte vector
// loads and stores, grid-stride over rows with a grid of a few CTAs per SM.
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

// dst[r] = (scale ? scale[p] : 1) * src[p / k], p = pair_of_row[r]; 0 if p is
// outside [0, P)
__global__ void __launch_bounds__(kThreads)
    permute_kernel(const uint4* __restrict__ src, const float* __restrict__ scale,
                   const int32_t* __restrict__ pair_of_row, int P, int k, int dv, int M_cap,
                   uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); r < M_cap;
       r += gridDim.x * kRowsPerBlock) {
    const int p = pair_of_row[r];
    uint4* out = dst + static_cast<long long>(r) * dv;
    if (p < 0 || p >= P) {
      for (int v = lane; v < dv; v += 32) out[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* in = src + static_cast<long long>(p / k) * dv;
    if (scale == nullptr) {
      int v = lane;
      for (; v + 96 < dv; v += 128) {
        const uint4 a = __ldg(in + v), b = __ldg(in + v + 32), c = __ldg(in + v + 64),
                    d = __ldg(in + v + 96);
        out[v] = a; out[v + 32] = b; out[v + 64] = c; out[v + 96] = d;
      }
      for (; v < dv; v += 32) out[v] = __ldg(in + v);
    } else {
      const float s = scale[p];
      for (int v = lane; v < dv; v += 32) out[v] = scale_bf16x8(__ldg(in + v), s);
    }
  }
}

// dst[t] = sum_j w_tj src[row(t,j)] (fp32, j ascending)
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const uint4* __restrict__ src, const float* __restrict__ probs,
                   const int32_t* __restrict__ row_of_pair, int T, int k, int dv, int M_cap,
                   uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); t < T;
       t += gridDim.x * kRowsPerBlock) {
    uint4* out = dst + static_cast<long long>(t) * dv;
    for (int v = lane; v < dv; v += 32) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int j = 0; j < k; ++j) {
        const int row = row_of_pair[t * k + j];
        if (row < 0 || row >= M_cap) continue;
        const float w = probs ? probs[t * k + j] : 1.0f;
        const uint4 y = __ldg(src + static_cast<long long>(row) * dv + v);
        const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(w, bf16_lo(yw[i]), acc[2 * i]);
          acc[2 * i + 1] = fmaf(w, bf16_hi(yw[i]), acc[2 * i + 1]);
        }
      }
      out[v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// dprobs[t*k+j] = <dO[t], src[row(t,j)]> (fp32; fixed per-lane order, then a
// fixed butterfly across lanes: deterministic)
__global__ void __launch_bounds__(kThreads)
    router_grad_kernel(const uint4* __restrict__ src, const uint4* __restrict__ dO,
                       const int32_t* __restrict__ row_of_pair, int T, int k, int dv, int M_cap,
                       float* __restrict__ dprobs) {
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); t < T;
       t += gridDim.x * kRowsPerBlock) {
    const uint4* g = dO + static_cast<long long>(t) * dv;
    for (int j = 0; j < k; ++j) {
      const int row = row_of_pair[t * k + j];
      float acc = 0.f;
      if (row >= 0 && row < M_cap) {
        const uint4* y = src + static_cast<long long>(row) * dv;
        for (int v = lane; v < dv; v += 32) {
          const uint4 a = __ldg(g + v), b = __ldg(y + v);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc = fmaf(bf16_lo(aw[i]), bf16_lo(bw[i]), acc);
            acc = fmaf(bf16_hi(aw[i]), bf16_hi(bw[i]), acc);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) dprobs[t * k + j] = acc;
    }
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

int grid_for(long long rows, int num_sms) {
  const long long want = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long cap = 8LL * num_sms;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_permute(const uint16_t* src, const float* scale, const int32_t* pair_of_row,
                           int T, int k, int d, int M_cap, uint16_t* dst, int num_sms,
                           cudaStream_t s) {
  if (M_cap <= 0) return cudaSuccess;
  permute_kernel<<<grid_for(M_cap, num_sms), kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(src), scale, pair_of_row, T * k, k, d / 8, M_cap,
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
  if (dst) {
    combine_kernel<<<grid_for(T, num_sms), kThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(src), probs, row_of_pair, T, k, d / 8, M_cap,
        reinterpret_cast<uint4*>(dst));
    ++*launches;
  }
  if (dprobs) {
    router_grad_kernel<<<grid_for(T, num_sms), kThreads, 0, s>>>(
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
