// act.cuh - gate nonlinearities of the gated expert MLP and their
// derivatives, shared by the bf16 and MXFP8 epilogues.
//   SwiGLU: phi(g) = g * sigmoid(g) (Swish on the gate side, times the up
//           projection) - [CuTe] "핵심 아이디어 / 구조 / 동작 방식".
//   GeGLU:  phi(g) = 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))), the
//           tanh approximation of GELU (Hendrycks & Gimpel).
#pragma once

#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + __expf(-g)); }
constexpr float kGeluC = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluA = 0.044715f;

template <int ACT>
__device__ __forceinline__ float gate_phi(float g) {
  if constexpr (ACT == MOE_ACT_SWIGLU) {
    return g * sigmoidf_(g);
  } else {
    const float z = kGeluC * (g + kGeluA * g * g * g);
    return 0.5f * g * (1.0f + tanhf(z));
  }
}
// phi and phi' together
template <int ACT>
__device__ __forceinline__ void gate_phi_dphi(float g, float& ph, float& dph) {
  if constexpr (ACT == MOE_ACT_SWIGLU) {
    const float s = sigmoidf_(g);
    ph = g * s;
    dph = s * (1.0f + g * (1.0f - s));
  } else {
    const float z = kGeluC * (g + kGeluA * g * g * g);
    const float th = tanhf(z);
    ph = 0.5f * g * (1.0f + th);
    dph = 0.5f * (1.0f + th) + 0.5f * g * (1.0f - th * th) * kGeluC * (1.0f + 3.0f * kGeluA * g * g);
  }
}

}  // namespace moe
