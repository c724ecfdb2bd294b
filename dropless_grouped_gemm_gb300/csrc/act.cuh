// act.cuh - gate nonlinearities of the gated expert MLP and their
// derivatives, shared by the bf16 and MXFP8 epilogues.
//   SwiGLU: phi(g) = g * sigmoid(g) (Swish on the gate side, times the up
//           projection) - [CuTe] "핵심 아이디어 / 구조 / 동작 방식".
//   GeGLU:  phi(g) = 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))), the
//           tanh approximation of GELU (Hendrycks & Gimpel), evaluated as
//           g sigmoid(2 sqrt(2/pi) (g + 0.044715 g^3)), the same function.
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
    // 1 + tanh(z) = 2 sigmoid(2z): no tanh, and no cancellation for
    // negative gates, where 1 + tanh(z) is small
    const float z = kGeluC * (g + kGeluA * g * g * g);
    return g * sigmoidf_(2.0f * z);
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
    // with s = sigmoid(2z): 1 + tanh z = 2s and 1 - tanh^2 z = 4 s (1 - s), so
    // phi = g s and phi' = s + 2 g s (1 - s) z'(g), z' = c (1 + 3 a g^2)
    const float z = kGeluC * (g + kGeluA * g * g * g);
    const float s = sigmoidf_(2.0f * z);
    ph = g * s;
    dph = s + 2.0f * g * s * (1.0f - s) * kGeluC * (1.0f + 3.0f * kGeluA * g * g);
  }
}

}  // namespace moe
