// act.cu - the expert MLP's activation and its derivative as separate
// memory passes over a stored H (and dA): the unfused form that the fused
// GEMM epilogues replace.  [CuTe] "무엇을 해결하려는가": without the fusion
// the activation is its own kernel that reads the FC1 output back from HBM
// and writes A, and the backward's derivative is another pass over dA and
// H.  The arithmetic is the epilogues' (act.cuh); the inputs are the bf16
// values those passes read back.
//
// HBM-bound: one thread takes 8 output columns of one row (16-byte vector
// accesses), grid-stride over the rows of every expert (rows at or past
// offsets[E] are not touched).
#include <cuda_runtime.h>

#include "act.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// A = act(H): gated rows hold (gate, up) pairs, A has half the columns
template <int ACT>
__global__ void __launch_bounds__(256)
    act_fwd_kernel(const uint16_t* __restrict__ h, const int32_t* __restrict__ offsets, int E,
                   long long rows_cap, int n, uint16_t* __restrict__ a) {
  const long long rows = min(static_cast<long long>(max(offsets[E], 0)), rows_cap);
  const int n8 = n / 8;
  const long long total = rows * n8;
  constexpr bool G = (ACT != MOE_ACT_SRELU);
  const int n1 = G ? 2 * n : n;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / n8;
    const int c8 = static_cast<int>(i - r * n8);
    uint32_t o[4];
    if constexpr (G) {
      const uint4* hp = reinterpret_cast<const uint4*>(h + r * n1 + 16 * c8);
      const uint4 v0 = hp[0], v1 = hp[1];
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a0 = gate_phi<ACT>(bf16_lo(w[2 * j])) * bf16_hi(w[2 * j]);
        const float a1 = gate_phi<ACT>(bf16_lo(w[2 * j + 1])) * bf16_hi(w[2 * j + 1]);
        o[j] = pack_bf16x2(a0, a1);
      }
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(h + r * n1 + 8 * c8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float h0 = fmaxf(bf16_lo(w[j]), 0.f), h1 = fmaxf(bf16_hi(w[j]), 0.f);
        o[j] = pack_bf16x2(h0 * h0, h1 * h1);
      }
    }
    *reinterpret_cast<uint4*>(a + r * n + 8 * c8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// dH = act'(H; dA): gated dg = dA u phi'(g), du = dA phi(g); sReLU
// dh = 2 max(h, 0) dA
template <int ACT>
__global__ void __launch_bounds__(256)
    act_bwd_kernel(const uint16_t* __restrict__ h, const uint16_t* __restrict__ da,
                   const int32_t* __restrict__ offsets, int E, long long rows_cap, int n,
                   uint16_t* __restrict__ dh) {
  const long long rows = min(static_cast<long long>(max(offsets[E], 0)), rows_cap);
  const int n8 = n / 8;
  const long long total = rows * n8;
  constexpr bool G = (ACT != MOE_ACT_SRELU);
  const int n1 = G ? 2 * n : n;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / n8;
    const int c8 = static_cast<int>(i - r * n8);
    const uint4 dv = *reinterpret_cast<const uint4*>(da + r * n + 8 * c8);
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
    if constexpr (G) {
      const uint4* hp = reinterpret_cast<const uint4*>(h + r * n1 + 16 * c8);
      const uint4 v0 = hp[0], v1 = hp[1];
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = (j & 1) ? bf16_hi(dw[j >> 1]) : bf16_lo(dw[j >> 1]);
        const float gg = bf16_lo(w[j]), uu = bf16_hi(w[j]);
        float ph, dph;
        gate_phi_dphi<ACT>(gg, ph, dph);
        o[j] = pack_bf16x2(d * uu * dph, d * ph);
      }
      uint4* op = reinterpret_cast<uint4*>(dh + r * n1 + 16 * c8);
      op[0] = make_uint4(o[0], o[1], o[2], o[3]);
      op[1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(h + r * n1 + 8 * c8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = pack_bf16x2(2.f * fmaxf(bf16_lo(w[j]), 0.f) * bf16_lo(dw[j]),
                           2.f * fmaxf(bf16_hi(w[j]), 0.f) * bf16_hi(dw[j]));
      *reinterpret_cast<uint4*>(dh + r * n1 + 8 * c8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

int grid_for(long long rows_cap, int n, int num_sms) {
  const long long want = (rows_cap * (n / 8) + 255) / 256;
  const long long most = 8LL * num_sms;
  return static_cast<int>(want < 1 ? 1 : (want < most ? want : most));
}

}  // namespace

cudaError_t launch_act_fwd(const uint16_t* h, const int32_t* offsets, int E, long long rows_cap,
                           int n, int act, uint16_t* a, int num_sms, cudaStream_t st) {
  const int grid = grid_for(rows_cap, n, num_sms);
  switch (act) {
    case MOE_ACT_SWIGLU: act_fwd_kernel<MOE_ACT_SWIGLU><<<grid, 256, 0, st>>>(h, offsets, E, rows_cap, n, a); break;
    case MOE_ACT_GEGLU: act_fwd_kernel<MOE_ACT_GEGLU><<<grid, 256, 0, st>>>(h, offsets, E, rows_cap, n, a); break;
    case MOE_ACT_SRELU: act_fwd_kernel<MOE_ACT_SRELU><<<grid, 256, 0, st>>>(h, offsets, E, rows_cap, n, a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_act_bwd(const uint16_t* h, const uint16_t* da, const int32_t* offsets, int E,
                           long long rows_cap, int n, int act, uint16_t* dh, int num_sms,
                           cudaStream_t st) {
  const int grid = grid_for(rows_cap, n, num_sms);
  switch (act) {
    case MOE_ACT_SWIGLU: act_bwd_kernel<MOE_ACT_SWIGLU><<<grid, 256, 0, st>>>(h, da, offsets, E, rows_cap, n, dh); break;
    case MOE_ACT_GEGLU: act_bwd_kernel<MOE_ACT_GEGLU><<<grid, 256, 0, st>>>(h, da, offsets, E, rows_cap, n, dh); break;
    case MOE_ACT_SRELU: act_bwd_kernel<MOE_ACT_SRELU><<<grid, 256, 0, st>>>(h, da, offsets, E, rows_cap, n, dh); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
