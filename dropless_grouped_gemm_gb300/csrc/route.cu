// route.cu - device-side routing layout: per-expert counts, ragged prefix
// offsets, and the stable pair <-> row maps of the expert-major buffer.
//
// [TE] "MoE 학습이 밀집 모델보다 어려운 이유: 래그드 텐서" and "최적화 1: grouped
// GEMM": the per-expert token counts are known only at run time and must stay
// on the device (no device-to-host copy, CUDA-graph capturable).
// [TE] ""드롭리스"의 실제 경계": expert-major rows, one per (token, expert)
// pair, each expert's region padded to the alignment unit; overflow past the
// buffer drops rows and reports the true total.
//
// Three kernels, all deterministic (every output is a function of the input
// alone; counting uses integer atomics only where order cannot matter):
//   1. route_hist:  chunk c of kChunk pairs -> ws[c][e] = #pairs of e in c
//   2. route_scan:  one block: exclusive prefix of ws over chunks (per e),
//                   counts, aligned offsets, true total, overflow flag
//   3. route_rank:  chunk c again, in pair order: stable rank of each pair
//                   among the pairs of its expert -> row_of_pair, pair_of_row
// pair_of_row is first filled with -1 (route_fill).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "ptx.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 16;
constexpr int kChunk = kThreads * kPerThread;  // 4096 pairs per chunk
constexpr int kWarps = kThreads / 32;

__global__ void route_fill(int32_t* __restrict__ p, int n, int32_t v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = v;
}

__global__ void __launch_bounds__(kThreads) route_hist(const int32_t* __restrict__ idx, int P, int E,
                                                       int32_t* __restrict__ ws,
                                                       int32_t* __restrict__ err) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kChunk;
  const int end = min(P, base + kChunk);
  bool bad = false;
  for (int p = base + threadIdx.x; p < end; p += kThreads) {
    const int e = idx[p];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else if (e != -1) bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_err(err, MOE_DEV_BAD_EXPERT);
  __syncthreads();
  int32_t* out = ws + static_cast<long long>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += kThreads) out[e] = hist[e];
}

// one block of 1024 threads; E <= 1024
__global__ void __launch_bounds__(1024) route_scan(int32_t* __restrict__ ws, int nchunks, int E,
                                                   int align, int M_cap,
                                                   int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ demanded,
                                                   int32_t* __restrict__ true_total,
                                                   int32_t* __restrict__ err) {
  __shared__ int32_t s_warp[32];
  const int e = threadIdx.x;
  int total_e = 0;
  if (e < E) {
    // exclusive prefix over chunks, in place
    for (int c = 0; c < nchunks; ++c) {
      int32_t* p = ws + static_cast<long long>(c) * E + e;
      const int v = *p;
      *p = total_e;
      total_e += v;
    }
    counts[e] = total_e;
  }
  // aligned count, block-wide exclusive scan over experts
  const long long aligned = (e < E) ? (static_cast<long long>(total_e) + align - 1) / align * align : 0;
  int v = static_cast<int>(aligned);  // T*k + E*align fits in int32 (checked on the host)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;  // exclusive warp base
  }
  __syncthreads();
  const int excl = s_warp[warp] + incl - v;
  if (e < E) {
    demanded[e] = excl;
    offsets[e] = min(excl, M_cap);
  }
  if (e == E - 1) {
    const int tot = excl + v;
    offsets[E] = min(tot, M_cap);
    *true_total = tot;
    if (tot > M_cap) set_err(err, MOE_DEV_OVERFLOW);
  }
}

__global__ void __launch_bounds__(kThreads) route_rank(const int32_t* __restrict__ idx, int P, int E,
                                                       int M_cap, const int32_t* __restrict__ ws,
                                                       const int32_t* __restrict__ demanded,
                                                       int32_t* __restrict__ row_of_pair,
                                                       int32_t* __restrict__ pair_of_row) {
  extern __shared__ int32_t sm[];
  int32_t* running = sm;            // [E] rows already given to e (chunk base + rounds)
  int32_t* wcnt = sm + E;           // [kWarps][E] per-round, per-warp counts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t* base_c = ws + static_cast<long long>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += kThreads) running[e] = demanded[e] + base_c[e];
  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * kChunk;
  for (int r = 0; r < kPerThread; ++r) {
    const int p = base + r * kThreads + threadIdx.x;
    int e = -1;
    if (p < P) {
      e = idx[p];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(mask) - 1;
    const int rank = __popc(mask & ((1u << lane) - 1u));
    if (e >= 0 && lane == leader) wcnt[warp * E + e] = __popc(mask);
    __syncthreads();
    int row = -1;
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += wcnt[w * E + e];
      row = running[e] + before + rank;
    }
    __syncthreads();
    if (e >= 0 && lane == leader) {
      atomicAdd(&running[e], __popc(mask));
      wcnt[warp * E + e] = 0;
    }
    if (p < P) {
      const int out = (row >= 0 && row < M_cap) ? row : -1;
      row_of_pair[p] = out;
      if (out >= 0) pair_of_row[out] = p;
    }
    __syncthreads();
  }
}

// Router: top-k experts of one token and the softmax of their logits, for
// one warp.  Lane l holds logits l, l+32, ..., NV of them (32 * NV >= E; the
// launchers take the smallest power of two, so that each round scans only
// the slots that can hold a logit).  Each of the k
// rounds takes the warp-wide largest logit not yet chosen, ties going to the
// lower expert index, so the choice is exact and deterministic.  Round j
// calls pick(j, expert, w) on every lane with the same values, w =
// exp(logit - top) unnormalised; returns the sum of the k weights.
// float -> 32-bit key whose unsigned order is the order of the floats (no
// NaN; -0 is keyed as +0, so that the two compare equal as floats do)
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NV, class Pick>
__device__ __forceinline__ float topk_warp(const float* __restrict__ row, int E, int k, int lane,
                                           Pick pick) {
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;
  float top = 0.f, sum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || bi == 0x7fffffff)) {
        bv = v[i];
        bi = e;
      }
    }
    // warp argmax in two reductions: the largest key, then the lowest
    // expert index among the lanes that hold it (0 marks a lane with no
    // candidate; every real key is above it)
    const uint32_t kv = (bi == 0x7fffffff) ? 0u : order_key(bv);
    const uint32_t km = __reduce_max_sync(0xffffffffu, kv);
    bi = static_cast<int>(__reduce_min_sync(
        0xffffffffu, (kv == km && bi != 0x7fffffff) ? static_cast<uint32_t>(bi) : 0xffffffffu));
    bv = key_value(km);
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) top = bv;
    const float ex = expf(bv - top);
    sum += ex;
    pick(j, bi, ex);
  }
  return sum;
}

// One warp per token: topk_idx and the normalised probabilities.
template <int NV>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                          int E, int k, int32_t* __restrict__ idx,
                                                          float* __restrict__ probs) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
    const long long p0 = static_cast<long long>(t) * k;
    const float sum = topk_warp<NV>(logits + static_cast<long long>(t) * E, E, k, lane,
                                [&](int j, int e, float w) {
                                  if (lane == 0) {
                                    idx[p0 + j] = e;
                                    probs[p0 + j] = w;   // normalised below
                                  }
                                });
    __syncwarp();
    for (int j = lane; j < k; j += 32) probs[p0 + j] /= sum;
  }
}

// The router fused into the routing layout's first pass ([TE] "Transformer
// Engine이 제공하는 세 가지 구성 요소": gate, top-k selection, dispatch and the
// grouped FFN in one fused block): the same selection as router_topk_kernel,
// and each chosen pair counted into its chunk's histogram ws[c][e] (c = pair
// / kChunk; ws is zeroed by route_fill2).  A block takes kTopkTokens
// consecutive tokens, one per warp, whose pairs lie in at most `rows`
// consecutive chunks (2 while kTopkTokens * k <= kChunk, 3 up to k = 1024):
// it counts them in shared memory and adds each non-zero count to ws with
// one atomic (a skewed router sends most tokens to a few experts, whose
// counters would otherwise take one global atomic per pair).  The counts
// are integer sums, so they do not depend on the order of the additions.
constexpr int kTopkTokens = 8;
template <int NV>
__global__ void __launch_bounds__(256) route_topk_hist(const float* __restrict__ logits, int T,
                                                       int E, int k, int32_t* __restrict__ idx,
                                                       float* __restrict__ probs,
                                                       int32_t* __restrict__ ws, int rows) {
  extern __shared__ int32_t hist[];   // [rows][E]: the block's first chunk and the next ones
  const int lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTopkTokens;
  const long long c0 = static_cast<long long>(t0) * k / kChunk;
  for (int i = threadIdx.x; i < rows * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int t = t0 + (threadIdx.x >> 5);
  if (t < T) {
    const long long p0 = static_cast<long long>(t) * k;
    const float sum = topk_warp<NV>(logits + static_cast<long long>(t) * E, E, k, lane,
                                [&](int j, int e, float w) {
                                  if (lane == 0) {
                                    idx[p0 + j] = e;
                                    probs[p0 + j] = w;
                                    atomicAdd(&hist[((p0 + j) / kChunk - c0) * E + e], 1);
                                  }
                                });
    __syncwarp();
    for (int j = lane; j < k; j += 32) probs[p0 + j] /= sum;
  }
  __syncthreads();
  // rows past the last chunk stay zero and are skipped
  for (int i = threadIdx.x; i < rows * E; i += blockDim.x) {
    const int v = hist[i];
    if (v != 0) atomicAdd(&ws[c0 * E + i], v);
  }
}

// pair_of_row <- -1 and, for the fused router, the chunk histograms <- 0
__global__ void route_fill2(int32_t* __restrict__ p, int n, int32_t* __restrict__ z, int nz) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n + nz; i += gridDim.x * blockDim.x) {
    if (i < n) p[i] = -1;
    else z[i - n] = 0;
  }
}

// logit slots per lane: the smallest power of two with 32 slots >= E
template <class F>
cudaError_t with_slots(int E, F&& f) {
  if (E <= 32) return f(std::integral_constant<int, 1>{});
  if (E <= 64) return f(std::integral_constant<int, 2>{});
  if (E <= 128) return f(std::integral_constant<int, 4>{});
  if (E <= 256) return f(std::integral_constant<int, 8>{});
  if (E <= 512) return f(std::integral_constant<int, 16>{});
  return f(std::integral_constant<int, 32>{});
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* idx,
                              float* probs, int num_sms, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const long long want = (static_cast<long long>(T) + 7) / 8;
  const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
  return with_slots(E, [&](auto nv) {
    router_topk_kernel<decltype(nv)::value><<<blocks, 256, 0, s>>>(logits, T, E, k, idx, probs);
    return cudaGetLastError();
  });
}

cudaError_t launch_route_logits(const float* logits, int T, int k, int E, int align, int M_cap,
                               int32_t* topk_idx, float* probs, int32_t* counts,
                               int32_t* offsets, int32_t* row_of_pair, int32_t* pair_of_row,
                               int32_t* true_total, void* workspace, int32_t* err, int num_sms,
                               cudaStream_t s, int* launches) {
  const int P = T * k;
  const int nchunks = (P + kChunk - 1) / kChunk;
  int32_t* ws = static_cast<int32_t*>(workspace);
  int32_t* demanded = ws + static_cast<long long>(nchunks) * E;
  *launches = 0;
  const long long nfill = static_cast<long long>(M_cap) + static_cast<long long>(nchunks) * E;
  if (nfill > 0) {
    const int blocks = static_cast<int>(min((nfill + 255) / 256, 4LL * num_sms));
    route_fill2<<<blocks, 256, 0, s>>>(pair_of_row, M_cap, ws, nchunks * E);
    ++*launches;
  }
  if (T > 0) {
    // the kTopkTokens * k pairs of a block's tokens touch at most `rows`
    // chunks (k <= E <= 1024: at most 12 KB of counters)
    const int rows = (kTopkTokens * k - 1) / kChunk + 2;
    const int blocks = (T + kTopkTokens - 1) / kTopkTokens;
    const cudaError_t e = with_slots(E, [&](auto nv) {
      route_topk_hist<decltype(nv)::value>
          <<<blocks, 32 * kTopkTokens, static_cast<size_t>(rows) * E * sizeof(int32_t), s>>>(
              logits, T, E, k, topk_idx, probs, ws, rows);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  route_scan<<<1, 1024, 0, s>>>(ws, nchunks, E, align, M_cap, counts, offsets, demanded,
                                true_total, err);
  ++*launches;
  if (nchunks > 0) {
    const size_t sm = static_cast<size_t>(E) * (1 + kWarps) * sizeof(int32_t);
    route_rank<<<nchunks, kThreads, sm, s>>>(topk_idx, P, E, M_cap, ws, demanded, row_of_pair,
                                             pair_of_row);
    ++*launches;
  }
  return cudaGetLastError();
}

size_t route_workspace_bytes(int T, int k, int E) {
  const long long P = static_cast<long long>(T) * k;
  const long long nchunks = (P + kChunk - 1) / kChunk;
  return static_cast<size_t>((nchunks * E + E) * sizeof(int32_t));
}

cudaError_t launch_route(const int32_t* topk_idx, int T, int k, int E, int align, int M_cap,
                         int32_t* counts, int32_t* offsets, int32_t* row_of_pair,
                         int32_t* pair_of_row, int32_t* true_total, void* workspace,
                         int32_t* err, int num_sms, cudaStream_t s, int* launches) {
  const int P = T * k;
  const int nchunks = (P + kChunk - 1) / kChunk;
  int32_t* ws = static_cast<int32_t*>(workspace);
  int32_t* demanded = ws + static_cast<long long>(nchunks) * E;
  *launches = 0;
  if (M_cap > 0) {
    const int blocks = min((M_cap + 255) / 256, 4 * num_sms);
    route_fill<<<blocks, 256, 0, s>>>(pair_of_row, M_cap, -1);
    ++*launches;
  }
  if (nchunks > 0) {
    route_hist<<<nchunks, kThreads, E * sizeof(int32_t), s>>>(topk_idx, P, E, ws, err);
    ++*launches;
  }
  route_scan<<<1, 1024, 0, s>>>(ws, nchunks, E, align, M_cap, counts, offsets, demanded,
                                true_total, err);
  ++*launches;
  if (nchunks > 0) {
    // at most (1 + 8) * 1024 * 4 = 36 KB: below the default 48 KB limit
    const size_t sm = static_cast<size_t>(E) * (1 + kWarps) * sizeof(int32_t);
    route_rank<<<nchunks, kThreads, sm, s>>>(topk_idx, P, E, M_cap, ws, demanded, row_of_pair,
                                             pair_of_row);
    ++*launches;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- no-alloc
// Scratch for callers that cannot allocate device memory: a fixed array in
// the library's own device image.  Every GPU that loads libmoe holds it
// (kRouteScratchWords * 4 bytes) until the process exits.  Host code must not
// pass the array's name to a kernel (on the host it is only a stand-in);
// the device address comes from cudaGetSymbolAddress, with the device
// current.  The address belongs to the module as loaded in one CUDA context,
// so it is cached per context: keyed by the context's unique ID
// (cuCtxGetId), which a context created later - e.g. the primary context
// that follows cudaDeviceReset - never reuses.
static __device__ __align__(256) int32_t g_route_scratch[kRouteScratchWords];

namespace {
std::mutex g_scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* ptr;
};
constexpr int kScratchCache = 64;
ScratchEntry g_scratch_cache[kScratchCache] = {};
int g_scratch_next = 0;

// unique ID of the calling thread's current context (0 if none or unknown)
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}
}  // namespace

cudaError_t route_scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = current_context_id();
  if (id != 0)
    for (const ScratchEntry& c : g_scratch_cache)
      if (c.ctx_id == id) {
        *out = c.ptr;
        return cudaSuccess;
      }
  // first call in this context (the lookup also brings up the device's
  // primary context when no context is current yet)
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
  if (e != cudaSuccess) return e;
  id = current_context_id();
  if (id != 0) {
    g_scratch_cache[g_scratch_next] = {id, p};
    g_scratch_next = (g_scratch_next + 1) % kScratchCache;
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace moe
