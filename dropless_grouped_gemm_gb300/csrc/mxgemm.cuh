// mxgemm.cuh - host-side interface of the MXFP8 kernels (mx.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

struct MxFc2Args {
  const int32_t* offsets;  // [E+1], multiples of 32
  int E;
  int M_cap;
  int n;                   // reduction length (multiple of 128)
  int d;                   // output columns (multiple of 128)
  const uint8_t* a_s;      // A row-wise scales, MMA-tiled by 32-row tile start
  const uint8_t* w2_s;     // W2 scales, MMA-tiled per expert
  uint16_t* out;           // y_perm [M_cap, d] bf16
  int32_t* err;
};

cudaError_t launch_mx_quantize_weights(const uint16_t* w2, int E, int n, int d, uint8_t* q,
                                       uint8_t* s, int num_sms, cudaStream_t st);
cudaError_t launch_mx_quantize_act(const uint16_t* src, int rows, int cols, const int32_t* offsets,
                                   int E, uint8_t* q, uint8_t* s, uint8_t* qT, uint8_t* sT,
                                   int32_t* err, int num_sms, cudaStream_t st);
cudaError_t launch_mx_fc2(const CUtensorMap& ta, const CUtensorMap& tb, const MxFc2Args& g,
                          int num_sms, cudaStream_t st);

}  // namespace moe
