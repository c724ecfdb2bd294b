// route.cuh - host-side interface of the routing-layout kernels (route.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

size_t route_workspace_bytes(int T, int k, int E);

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* idx,
                              float* probs, int num_sms, cudaStream_t s);

// Fixed scratch of the no-allocation routing entry point: 1 MiB.
constexpr size_t kRouteScratchWords = 262144;

// Device address of that scratch on the current device (looked up once per
// device, then cached).
cudaError_t route_scratch_address(void** out);

// Enqueues the routing-layout kernels; *launches receives their number.
cudaError_t launch_route(const int32_t* topk_idx, int T, int k, int E, int align, int M_cap,
                         int32_t* counts, int32_t* offsets, int32_t* row_of_pair,
                         int32_t* pair_of_row, int32_t* true_total, void* workspace,
                         int32_t* err, int num_sms, cudaStream_t s, int* launches);

// The router fused into the layout: top-k selection and softmax from the
// logits [T, E] (writes topk_idx and probs) inside the layout's first pass,
// then the same offsets and maps as launch_route.
cudaError_t launch_route_logits(const float* logits, int T, int k, int E, int align, int M_cap,
                                int32_t* topk_idx, float* probs, int32_t* counts,
                                int32_t* offsets, int32_t* row_of_pair, int32_t* pair_of_row,
                                int32_t* true_total, void* workspace, int32_t* err, int num_sms,
                                cudaStream_t s, int* launches);

cudaError_t launch_permute(const uint16_t* src, const float* scale, const int32_t* pair_of_row,
                           int T, int k, int d, int M_cap, uint16_t* dst, int num_sms,
                           cudaStream_t s);

// the same copy in token order from both (mutually inverse) maps, pad rows
// zeroed
cudaError_t launch_permute_tokens(const uint16_t* src, const float* scale,
                                  const int32_t* row_of_pair, const int32_t* pair_of_row, int T,
                                  int k, int d, int M_cap, uint16_t* dst, int num_sms,
                                  cudaStream_t s);

cudaError_t launch_unpermute(const uint16_t* src, const float* probs,
                             const int32_t* row_of_pair, int T, int k, int d, int M_cap,
                             uint16_t* dst,
                             const uint16_t* dO, float* dprobs, int num_sms, cudaStream_t s,
                             int* launches);

// dprobs[p] from the routed backward's per-row partials ds_part [M_cap, n_parts]
cudaError_t launch_router_grad_rows(const float* ds_part, int n_parts, const int32_t* row_of_pair,
                                   int P, int M_cap, float* dprobs, int num_sms, cudaStream_t s);

}  // namespace moe
