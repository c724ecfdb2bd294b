// api.cu - the extern "C" entry points of libmoe (declared in include/moe.h):
// host-side argument checks, TMA tensor-map encoding, launch sequencing.
// What each entry point computes, and the passage of the pages that defines
// it, is stated at its declaration in include/moe.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe.h"
#include "gemm.cuh"
#include "mxgemm.cuh"
#include "route.cuh"

namespace moe {
cudaError_t launch_bounded_wait_selftest(int limit_us, int32_t* err, int32_t* waited_us,
                                         cudaStream_t s);
}  // namespace moe

namespace {

thread_local int g_last_launches = 0;
// kernels beyond one that launch_grouped_gemm made for a call (a skinny
// layer's GEMM splits its hot experts into a launch of their own)
thread_local int g_split_extra = 0;
thread_local cudaEvent_t const* g_events = nullptr;
thread_local int g_events_n = 0;
thread_local int g_events_used = 0;

// measurement hook: events around one launch (or one whole call)
void ev_begin(cudaStream_t s) {
  if (g_events && g_events_used + 1 < g_events_n) cudaEventRecord(g_events[g_events_used], s);
}
void ev_end(cudaStream_t s) {
  if (g_events && g_events_used + 1 < g_events_n) {
    cudaEventRecord(g_events[g_events_used + 1], s);
    g_events_used += 2;
  }
}
cudaError_t gemm(moe::GemmKind kind, int act, const CUtensorMap& ta, const CUtensorMap& tb,
                 const CUtensorMap& tc, const moe::GemmArgs& g, int sms, cudaStream_t s,
                 const CUtensorMap* td = nullptr) {
  ev_begin(s);
  int launched = 1;
  const cudaError_t e =
      moe::launch_grouped_gemm(kind, act, ta, tb, tc, g, sms, s, false, td, &launched);
  g_split_extra += launched - 1;
  ev_end(s);
  return e;
}

cudaError_t mx_gemm(moe::MxKind kind, int act, const CUtensorMap& ta, const CUtensorMap& tb,
                    const CUtensorMap& tc, const moe::MxGemmArgs& g, int sms, cudaStream_t s) {
  ev_begin(s);
  int launched = 1;
  const cudaError_t e = moe::launch_mx_gemm(kind, act, ta, tb, tc, g, sms, s, &launched);
  g_split_extra += launched - 1;
  ev_end(s);
  return e;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// 256-byte aligned carving of a caller-provided workspace
struct Carve {
  uint8_t* base;
  size_t used;
  uint8_t* take(size_t bytes) {
    uint8_t* p = base ? base + used : nullptr;
    used += (bytes + 255) & ~static_cast<size_t>(255);
    return p;
  }
};

// regions of the MXFP8 backward's workspace, in carving order
struct MxBwdWs {
  uint8_t *dy_q, *dy_s, *dy_qT, *dy_sT, *x_qT, *x_sT, *a_sT, *dh_q, *dh_s, *dh_qT, *dh_sT;
  size_t bytes;
};
MxBwdWs carve_mx_bwd(void* base, int M_cap, int d, int n1, int n) {
  Carve c{static_cast<uint8_t*>(base), 0};
  const size_t M = static_cast<size_t>(M_cap);
  MxBwdWs w;
  w.dy_q = c.take(M * d);
  w.dy_s = c.take(M * d / 8);
  w.dy_qT = c.take(M * d);
  w.dy_sT = c.take(M * d / 8);
  w.x_qT = c.take(M * d);
  w.x_sT = c.take(M * d / 8);
  w.a_sT = c.take(M * n / 8);
  w.dh_q = c.take(M * n1);
  w.dh_s = c.take(M * n1 / 8);
  w.dh_qT = c.take(M * n1);
  w.dh_sT = c.take(M * n1 / 8);
  w.bytes = c.used;
  return w;
}

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// tensor map (bf16 or u8), 128-byte swizzle; dims/box listed innermost first.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint32_t* box, bool u8 = false,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t bdim[3], estr[3] = {1, 1, 1};
  uint64_t stride = u8 ? 1 : 2;
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  const CUresult r = fn(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        rank, const_cast<void*>(base), gdim,
                        gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [rows, cols] activation matrix, box (128 bytes of cols) x (box_rows rows)
bool map_act(CUtensorMap* m, const void* p, int rows, int cols, int box_rows, bool u8 = false) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint32_t box[2] = {u8 ? 128u : 64u, static_cast<uint32_t>(box_rows)};
  return make_map(m, p, 2, dims, box, u8);
}
// [E, rows, cols] weights, box (128 bytes of cols) x (box_rows rows) x 1
bool map_w(CUtensorMap* m, const void* p, int E, int rows, int cols, int box_rows,
           bool u8 = false) {
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(E)};
  const uint32_t box[3] = {u8 ? 128u : 64u, static_cast<uint32_t>(box_rows), 1};
  return make_map(m, p, 3, dims, box, u8);
}

// [E, rows, cols] bf16 output written by staged TMA stores: box (64 cols,
// 128-byte swizzle) or (32 cols, 64-byte swizzle) x 32 rows x 1
bool map_out3(CUtensorMap* m, const void* p, int E, int rows, int cols, bool wide) {
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(E)};
  const uint32_t box[3] = {wide ? 64u : 32u, 32, 1};
  return make_map(m, p, 3, dims, box, false,
                  wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// [rows, cols] bf16 output written by staged TMA stores of FC2 / FC1-dgrad:
// box 32 cols x 32 rows, 64-byte swizzle
bool map_out2(CUtensorMap* m, const void* p, int rows, int cols) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint32_t box[2] = {32, 32};
  return make_map(m, p, 2, dims, box, false, CU_TENSOR_MAP_SWIZZLE_64B);
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_E_CUDA; }

int check_mlp_sizes(int E, int M_cap, int d, int n) {
  if (E < 1 || E > MOE_MAX_EXPERTS) return MOE_E_SIZE;
  if (M_cap < 0 || d <= 0 || n <= 0 || d % 64 || n % 64) return MOE_E_SIZE;
  if (static_cast<long long>(M_cap) * 2 * n >= (1LL << 40)) return MOE_E_SIZE;
  return MOE_OK;
}

// The four backward GEMMs.  dy is FC2-dgrad's A operand and FC2-wgrad's B
// operand, a_w FC2-wgrad's A operand.  Routed (probs != NULL): dy is the
// unscaled gathered dO; FC2-dgrad applies each row's router probability in
// its epilogue, which also writes A' (= a_w) and the dS partials.  With
// x_tok / do_tok (routed only) the token tensors x [T, d] and dO [T, d]
// replace x_perm and dy: the GEMMs read their rows through pair_of_row.
int bwd_gemms(const moe_bf16* x_perm, const moe_bf16* h_saved, const moe_bf16* a_w,
              const moe_bf16* dy, const int32_t* offsets, int E, int M_cap, int d, int n,
              const moe_bf16* W1, const moe_bf16* W2, int act, moe_bf16* dh, moe_bf16* dx_perm,
              moe_bf16* dW1, moe_bf16* dW2, int32_t* err, cudaStream_t s, int sms,
              const int32_t* pair_of_row, const float* probs, moe_bf16* a_scaled,
              float* ds_part, float* amax_dh, bool accumulate,
              const moe_bf16* x_tok = nullptr, const moe_bf16* do_tok = nullptr, int T = 0,
              int k = 1) {
  const bool gather = x_tok != nullptr;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  moe::GemmArgs probe{};
  probe.M_cap = M_cap;
  probe.E = E;
  const bool skinny = moe::wgrad_skinny(probe);
  // operand maps
  CUtensorMap t_dy_k, t_w2_k, t_a_mn, t_dy_mn, t_dh_k, t_w1_k, t_x_mn, t_dh_mn, t_dw1, t_dw2;
  if (!map_act(&t_dy_k, dy, M_cap, d, moe::kBM) ||           // FC2-dgrad A (K = d)
      !map_w(&t_w2_k, W2, E, n, d, 128) ||                    // FC2-dgrad B rows = n (halves)
      !map_act(&t_a_mn, a_w, M_cap, n, 64) ||                 // FC2-wgrad A (MN = n)
      !map_act(&t_dy_mn, dy, M_cap, d, 64) ||                 // FC2-wgrad B (MN = d)
      !map_act(&t_dh_k, dh, M_cap, n1, moe::kBM) ||           // FC1-dgrad A (K = n1)
      !map_w(&t_w1_k, W1, E, d, n1, 128) ||                   // FC1-dgrad B rows = d (halves)
      !map_act(&t_x_mn, x_perm, M_cap, d, 64) ||              // FC1-wgrad A (MN = d)
      !map_act(&t_dh_mn, dh, M_cap, n1, 64) ||                // FC1-wgrad B (MN = n1)
      !map_out3(&t_dw2, dW2, E, n, d, skinny) || !map_out3(&t_dw1, dW1, E, d, n1, skinny))
    return MOE_E_CUDA;
  // gathered: FC2-dgrad's A and FC2-wgrad's B are dO's rows, FC1-wgrad's A
  // x's rows (the maps built above on the token tensors go unused)
  auto set_gather = [&](moe::GemmArgs& ga, int operand, const moe_bf16* src) {
    if (!gather) return;
    ga.gather_pair = pair_of_row; ga.gather_k = k; ga.gather_T = T;
    ga.gather_operand = operand; ga.gather_src = src; ga.gather_ld = d;
  };

  // 1. dH = act'(H; dY W2^T)
  moe::GemmArgs g{};
  g.offsets = offsets; g.E = E; g.M_cap = M_cap; g.K = d; g.N = n;
  g.out = dh; g.ldo = n1; g.aux = h_saved; g.ld_aux = n1; g.err = err; g.amax = amax_dh;
  if (probs) {
    g.pair_of_row = pair_of_row; g.probs = probs; g.out3 = a_scaled; g.ldo3 = n;
    g.ds_part = ds_part; g.ds_parts = (n + 127) / 128;
  }
  set_gather(g, 0, do_tok);
  // dH (and A') leave through staged TMA stores
  CUtensorMap t_dh_o, t_as_o = t_dy_k;
  if (!map_out2(&t_dh_o, dh, M_cap, n1) || (probs && !map_out2(&t_as_o, a_scaled, M_cap, n)))
    return MOE_E_CUDA;
  g.tma_out = 1;
  cudaError_t e = gemm(moe::GemmKind::kDgradAct, act, t_dy_k, t_w2_k, t_dh_o, g, sms, s, &t_as_o);
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 2. dW2_e = A_e^T dY_e
  moe::GemmArgs gw2{};
  gw2.offsets = offsets; gw2.E = E; gw2.M_cap = M_cap; gw2.N = d; gw2.R = n;
  gw2.out = dW2; gw2.ldo = d; gw2.out_estride = static_cast<long long>(n) * d; gw2.err = err;
  gw2.accumulate = accumulate;
  set_gather(gw2, 1, do_tok);
  // a skinny layer's hot experts run with the large-expert staging: its box
  CUtensorMap t_dw2_l, t_dw1_l;
  if (skinny && (!map_out3(&t_dw2_l, dW2, E, n, d, false) || !map_out3(&t_dw1_l, dW1, E, d, n1, false)))
    return MOE_E_CUDA;
  e = gemm(moe::GemmKind::kWgrad, 0, t_a_mn, t_dy_mn, t_dw2, gw2, sms, s, skinny ? &t_dw2_l : nullptr);
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 3. dX = dH W1^T
  moe::GemmArgs gd{};
  gd.offsets = offsets; gd.E = E; gd.M_cap = M_cap; gd.K = n1; gd.N = d;
  gd.out = dx_perm; gd.ldo = d; gd.err = err;
  CUtensorMap t_dx;
  if (!map_out2(&t_dx, dx_perm, M_cap, d)) return MOE_E_CUDA;
  gd.tma_out = 1;
  e = gemm(moe::GemmKind::kDgrad, 0, t_dh_k, t_w1_k, t_dx, gd, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 4. dW1_e = X_e^T dH_e
  moe::GemmArgs gw1{};
  gw1.offsets = offsets; gw1.E = E; gw1.M_cap = M_cap; gw1.N = n1; gw1.R = d;
  gw1.out = dW1; gw1.ldo = n1; gw1.out_estride = static_cast<long long>(d) * n1; gw1.err = err;
  gw1.accumulate = accumulate;
  set_gather(gw1, 0, x_tok);
  e = gemm(moe::GemmKind::kWgrad, 0, t_x_mn, t_dh_mn, t_dw1, gw1, sms, s, skinny ? &t_dw1_l : nullptr);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = 4 + g_split_extra;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_version(void) { return "libmoe 0.1.0 (sm_103a, tcgen05/TMA grouped GEMM)"; }

int moe_last_launch_count(void) { return g_last_launches; }

int moe_selftest_bounded_wait(int limit_us, int32_t* err, int32_t* waited_us, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (limit_us < 1 || limit_us > 1000000) return MOE_E_SIZE;
  if (!err || !waited_us) return MOE_E_NULL;
  const cudaError_t e = moe::launch_bounded_wait_selftest(limit_us, err, waited_us,
                                                          static_cast<cudaStream_t>(stream));
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

int moe_set_launch_events(void* const* events, int n) {
  g_events = reinterpret_cast<cudaEvent_t const*>(events);
  g_events_n = (events && n > 0) ? n : 0;
  if (!g_events_n) g_events = nullptr;
  g_events_used = 0;
  return MOE_OK;
}

int moe_launch_events_used(void) { return g_events_used; }

int moe_router_topk(const float* logits, int T, int E, int k, int32_t* topk_idx, float* probs,
                    void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E) return MOE_E_SIZE;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !probs) return MOE_E_NULL;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_router_topk(logits, T, E, k, topk_idx, probs, sms, s);
  ev_end(s);
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

size_t moe_route_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return moe::route_workspace_bytes(T, k, E);
}

int moe_route_offsets(const int32_t* topk_idx, int T, int k, int E, int align, int M_cap,
                      int32_t* counts, int32_t* offsets, int32_t* row_of_pair,
                      int32_t* pair_of_row, int32_t* true_total, void* workspace,
                      size_t ws_bytes, int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || E < 1 || E > MOE_MAX_EXPERTS || k > E || align < 1 || align > 4096 ||
      M_cap < 0)
    return MOE_E_SIZE;
  if (static_cast<long long>(T) * k + static_cast<long long>(E) * align >= (1LL << 31))
    return MOE_E_SIZE;
  if (!counts || !offsets || !true_total || !err) return MOE_E_NULL;
  if (T > 0 && (!topk_idx || !row_of_pair)) return MOE_E_NULL;
  if (M_cap > 0 && !pair_of_row) return MOE_E_NULL;
  if (ws_bytes < moe::route_workspace_bytes(T, k, E)) return MOE_E_WORKSPACE;
  if (!workspace) return MOE_E_NULL;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  int launches = 0;
  ev_begin(static_cast<cudaStream_t>(stream));
  const cudaError_t e = moe::launch_route(topk_idx, T, k, E, align, M_cap, counts, offsets,
                                          row_of_pair, pair_of_row, true_total, workspace, err,
                                          sms, static_cast<cudaStream_t>(stream), &launches);
  ev_end(static_cast<cudaStream_t>(stream));
  g_last_launches = launches + g_split_extra;
  return cuda_rc(e);
}

int moe_route_logits(const float* logits, int T, int E, int k, int align, int M_cap,
                     int32_t* topk_idx, float* probs, int32_t* counts, int32_t* offsets,
                     int32_t* row_of_pair, int32_t* pair_of_row, int32_t* true_total,
                     void* workspace, size_t ws_bytes, int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || E < 1 || E > MOE_MAX_EXPERTS || k > E || align < 1 || align > 4096 ||
      M_cap < 0)
    return MOE_E_SIZE;
  if (static_cast<long long>(T) * k + static_cast<long long>(E) * align >= (1LL << 31))
    return MOE_E_SIZE;
  if (!counts || !offsets || !true_total || !err) return MOE_E_NULL;
  if (T > 0 && (!logits || !topk_idx || !probs || !row_of_pair)) return MOE_E_NULL;
  if (M_cap > 0 && !pair_of_row) return MOE_E_NULL;
  if (ws_bytes < moe::route_workspace_bytes(T, k, E)) return MOE_E_WORKSPACE;
  if (!workspace) return MOE_E_NULL;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  int launches = 0;
  ev_begin(static_cast<cudaStream_t>(stream));
  const cudaError_t e = moe::launch_route_logits(logits, T, k, E, align, M_cap, topk_idx, probs,
                                                 counts, offsets, row_of_pair, pair_of_row,
                                                 true_total, workspace, err, sms,
                                                 static_cast<cudaStream_t>(stream), &launches);
  ev_end(static_cast<cudaStream_t>(stream));
  g_last_launches = launches + g_split_extra;
  return cuda_rc(e);
}

int moe_route_offsets_noalloc(const int32_t* topk_idx, int T, int k, int E, int align, int M_cap,
                              int32_t* counts, int32_t* offsets, int32_t* row_of_pair,
                              int32_t* pair_of_row, int32_t* true_total, int32_t* err,
                              void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || E < 1 || E > MOE_MAX_EXPERTS || k > E || align < 1 || align > 4096 ||
      M_cap < 0)
    return MOE_E_SIZE;
  if (static_cast<long long>(T) * k + static_cast<long long>(E) * align >= (1LL << 31))
    return MOE_E_SIZE;
  if (moe::route_workspace_bytes(T, k, E) > moe::kRouteScratchWords * sizeof(int32_t))
    return MOE_E_WORKSPACE;  // needs more than the fixed scratch holds
  if (!counts || !offsets || !true_total || !err) return MOE_E_NULL;
  if (T > 0 && (!topk_idx || !row_of_pair)) return MOE_E_NULL;
  if (M_cap > 0 && !pair_of_row) return MOE_E_NULL;
  void* scratch = nullptr;
  if (moe::route_scratch_address(&scratch) != cudaSuccess || scratch == nullptr)
    return MOE_E_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  int launches = 0;
  ev_begin(static_cast<cudaStream_t>(stream));
  const cudaError_t e = moe::launch_route(topk_idx, T, k, E, align, M_cap, counts, offsets,
                                          row_of_pair, pair_of_row, true_total, scratch, err,
                                          sms, static_cast<cudaStream_t>(stream), &launches);
  ev_end(static_cast<cudaStream_t>(stream));
  g_last_launches = launches + g_split_extra;
  return cuda_rc(e);
}

int moe_permute(const moe_bf16* src, const float* scale, const int32_t* pair_of_row, int T, int k,
                int d, int M_cap, moe_bf16* dst, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || d <= 0 || d % 64 || M_cap < 0) return MOE_E_SIZE;
  if (M_cap == 0) return MOE_OK;
  if (!pair_of_row || !dst || (T > 0 && !src)) return MOE_E_NULL;
  if (misaligned(src) || misaligned(dst)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  ev_begin(static_cast<cudaStream_t>(stream));
  const cudaError_t e = moe::launch_permute(src, scale, pair_of_row, T, k, d, M_cap, dst, sms,
                                            static_cast<cudaStream_t>(stream));
  ev_end(static_cast<cudaStream_t>(stream));
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

int moe_permute_tokens(const moe_bf16* src, const float* scale, const int32_t* row_of_pair,
                       const int32_t* pair_of_row, int T, int k, int d, int M_cap, moe_bf16* dst,
                       void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || d <= 0 || d % 64 || M_cap < 0) return MOE_E_SIZE;
  if (static_cast<long long>(T) * k >= (1LL << 31)) return MOE_E_SIZE;
  if (M_cap == 0) return MOE_OK;
  if (!pair_of_row || !dst || (T > 0 && (!src || !row_of_pair))) return MOE_E_NULL;
  if (misaligned(src) || misaligned(dst)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  ev_begin(static_cast<cudaStream_t>(stream));
  const cudaError_t e = moe::launch_permute_tokens(src, scale, row_of_pair, pair_of_row, T, k, d,
                                                   M_cap, dst, sms,
                                                   static_cast<cudaStream_t>(stream));
  ev_end(static_cast<cudaStream_t>(stream));
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

int moe_unpermute(const moe_bf16* src, const float* probs, const int32_t* row_of_pair, int T,
                  int k, int d, int M_cap, moe_bf16* dst, const moe_bf16* dO, float* dprobs,
                  void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || d <= 0 || d % 64 || M_cap < 0) return MOE_E_SIZE;
  if (T == 0) return MOE_OK;
  if (!src || !row_of_pair) return MOE_E_NULL;
  if (!dst && !dprobs) return MOE_E_NULL;
  if (dprobs && !dO) return MOE_E_NULL;
  if (misaligned(src) || misaligned(dst) || misaligned(dO)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  int launches = 0;
  ev_begin(static_cast<cudaStream_t>(stream));
  const cudaError_t e = moe::launch_unpermute(src, probs, row_of_pair, T, k, d, M_cap, dst, dO,
                                              dprobs, sms, static_cast<cudaStream_t>(stream),
                                              &launches);
  ev_end(static_cast<cudaStream_t>(stream));
  g_last_launches = launches + g_split_extra;
  return cuda_rc(e);
}

int moe_grouped_mlp_fwd(const moe_bf16* x_perm, const int32_t* offsets, int E, int M_cap, int d,
                        int n, const moe_bf16* W1, const moe_bf16* W2, int act, int flags,
                        moe_bf16* h_saved, moe_bf16* a, moe_bf16* y_perm, const moe_mx_fwd* mx,
                        float* amax_a, int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, d, n);
  if (rc) return rc;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU ||
      (flags & ~(MOE_FLAG_SAVE_H | MOE_FLAG_MXFP8)))
    return MOE_E_ARG;
  const bool save_h = flags & MOE_FLAG_SAVE_H;
  const bool use_mx = flags & MOE_FLAG_MXFP8;
  if (use_mx) {
    if (!mx || !mx->w2_q || !mx->w2_s || !mx->a_q || !mx->a_s || (mx->a_qT && !mx->a_sT) ||
        (mx->y_q && !mx->y_s))
      return MOE_E_NULL;
    if (misaligned(mx->y_q)) return MOE_E_ALIGN;
    if (n % 128 || d % 128 || M_cap % 32) return MOE_E_SIZE;
    if (misaligned(mx->w2_q) || misaligned(mx->w2_s) || misaligned(mx->a_q) ||
        misaligned(mx->a_s) || misaligned(mx->a_qT))
      return MOE_E_ALIGN;
  }
  if (!offsets || !W1 || (!W2 && !use_mx) || !err) return MOE_E_NULL;
  if (M_cap == 0) return MOE_OK;
  if (!x_perm || !a || !y_perm || (save_h && !h_saved)) return MOE_E_NULL;
  if (misaligned(x_perm) || misaligned(W1) || misaligned(W2) || misaligned(a) ||
      misaligned(y_perm) || (save_h && misaligned(h_saved)))
    return MOE_E_ALIGN;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tx, tw1, ta, tw2;
  if (!map_act(&tx, x_perm, M_cap, d, moe::kBM) || !map_w(&tw1, W1, E, d, n1, 64))
    return MOE_E_CUDA;
  if (use_mx) {
    if (!map_act(&ta, mx->a_q, M_cap, n, 128, true) || !map_w(&tw2, mx->w2_q, E, n, d, 128, true))
      return MOE_E_CUDA;
  } else if (!map_act(&ta, a, M_cap, n, moe::kBM) || !map_w(&tw2, W2, E, n, d, 64)) {
    return MOE_E_CUDA;
  }
  moe::GemmArgs g1{};
  g1.offsets = offsets; g1.E = E; g1.M_cap = M_cap; g1.K = d; g1.N = n1; g1.R = 0;
  g1.out = a; g1.ldo = n; g1.out2 = save_h ? h_saved : nullptr; g1.ldo2 = n1; g1.err = err;
  g1.amax = amax_a;
  if (use_mx) {
    g1.mx_q = mx->a_q; g1.mx_s = mx->a_s; g1.mx_qT = mx->a_qT;
    g1.mx_sT = mx->a_qT ? mx->a_sT : nullptr; g1.n_a = n;
  }
  // H and A leave through staged TMA stores (with MXFP8 outputs, the
  // transposed copy goes through the same staging box)
  CUtensorMap th = tx, tao = tx;
  if ((save_h && !map_out2(&th, h_saved, M_cap, n1)) || !map_out2(&tao, a, M_cap, n))
    return MOE_E_CUDA;
  g1.tma_out = 1;
  ev_begin(s);
  int launched = 1;
  cudaError_t e = moe::launch_grouped_gemm(moe::GemmKind::kFc1Act, act, tx, tw1, th, g1, sms, s,
                                           use_mx, &tao, &launched);
  g_split_extra += launched - 1;
  ev_end(s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  if (use_mx) {
    moe::MxGemmArgs q{};
    q.offsets = offsets; q.E = E; q.M_cap = M_cap; q.K = n; q.N = d;
    q.a_s = mx->a_s; q.b_s = mx->w2_s; q.out = y_perm; q.ldo = d; q.err = err;
    // scale sizes: A's row tiles, W2's column tiles (for the pair mode's TMA)
    q.a_s_bytes = static_cast<long long>(M_cap) * n / 8;
    q.b_s_bytes = static_cast<long long>(E) * n * d / 32;
    q.q_out = mx->y_q; q.s_out = mx->y_q ? mx->y_s : nullptr;
    CUtensorMap ty;
    if (!map_out2(&ty, y_perm, M_cap, d)) return MOE_E_CUDA;
    q.tma_out = 1;
    ev_begin(s);
    e = moe::launch_mx_gemm(moe::MxKind::kFc2, 0, ta, tw2, ty, q, sms, s);
    ev_end(s);
    if (e != cudaSuccess) return MOE_E_CUDA;
    g_last_launches = 2 + g_split_extra;
    return MOE_OK;
  }
  moe::GemmArgs g2{};
  g2.offsets = offsets; g2.E = E; g2.M_cap = M_cap; g2.K = n; g2.N = d; g2.R = 0;
  g2.out = y_perm; g2.ldo = d; g2.err = err;
  CUtensorMap ty;
  if (!map_out2(&ty, y_perm, M_cap, d)) return MOE_E_CUDA;
  g2.tma_out = 1;
  e = gemm(moe::GemmKind::kFc2, 0, ta, tw2, ty, g2, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = 2 + g_split_extra;
  return MOE_OK;
}

int moe_grouped_mlp_bwd(const moe_bf16* x_perm, const moe_bf16* h_saved, const moe_bf16* a,
                        const moe_bf16* dy_perm, const int32_t* offsets, int E, int M_cap, int d,
                        int n, const moe_bf16* W1, const moe_bf16* W2, int act, int flags,
                        moe_bf16* dh, moe_bf16* dx_perm, moe_bf16* dW1, moe_bf16* dW2,
                        float* amax_dh, int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, d, n);
  if (rc) return rc;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU || (flags & ~MOE_FLAG_ACCUMULATE_DW))
    return MOE_E_ARG;
  const bool accumulate = flags & MOE_FLAG_ACCUMULATE_DW;
  if (!offsets || !W1 || !W2 || !dW1 || !dW2 || !err) return MOE_E_NULL;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M_cap == 0) {
    // no rows at all: the weight gradients are exactly zero (untouched
    // when accumulating)
    if (accumulate) return MOE_OK;
    cudaError_t e = cudaMemsetAsync(dW1, 0, static_cast<size_t>(E) * d * n1 * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, static_cast<size_t>(E) * n * d * 2, s);
    return cuda_rc(e);
  }
  if (!x_perm || !h_saved || !a || !dy_perm || !dh || !dx_perm) return MOE_E_NULL;
  if (misaligned(x_perm) || misaligned(h_saved) || misaligned(a) || misaligned(dy_perm) ||
      misaligned(dh) || misaligned(dx_perm) || misaligned(dW1) || misaligned(dW2) ||
      misaligned(W1) || misaligned(W2))
    return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;

  return bwd_gemms(x_perm, h_saved, a, dy_perm, offsets, E, M_cap, d, n, W1, W2, act, dh, dx_perm,
                   dW1, dW2, err, s, sms, nullptr, nullptr, nullptr, nullptr, amax_dh, accumulate);
}

int moe_grouped_mlp_bwd_routed(const moe_bf16* x_perm, const moe_bf16* h_saved,
                               const moe_bf16* do_perm, const int32_t* pair_of_row,
                               const float* probs, const int32_t* offsets, int E, int M_cap,
                               int d, int n, const moe_bf16* W1, const moe_bf16* W2, int act,
                               int flags, moe_bf16* dh, moe_bf16* a_scaled, float* ds_part,
                               moe_bf16* dx_perm, moe_bf16* dW1, moe_bf16* dW2, float* amax_dh,
                               int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, d, n);
  if (rc) return rc;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU || (flags & ~MOE_FLAG_ACCUMULATE_DW))
    return MOE_E_ARG;
  const bool accumulate = flags & MOE_FLAG_ACCUMULATE_DW;
  if (!offsets || !W1 || !W2 || !dW1 || !dW2 || !err) return MOE_E_NULL;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M_cap == 0) {
    if (accumulate) return MOE_OK;
    cudaError_t e = cudaMemsetAsync(dW1, 0, static_cast<size_t>(E) * d * n1 * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, static_cast<size_t>(E) * n * d * 2, s);
    return cuda_rc(e);
  }
  if (!x_perm || !h_saved || !do_perm || !pair_of_row || !probs || !dh || !a_scaled || !ds_part ||
      !dx_perm)
    return MOE_E_NULL;
  if (misaligned(x_perm) || misaligned(h_saved) || misaligned(do_perm) || misaligned(dh) ||
      misaligned(a_scaled) || misaligned(dx_perm) || misaligned(dW1) || misaligned(dW2) ||
      misaligned(W1) || misaligned(W2))
    return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  return bwd_gemms(x_perm, h_saved, a_scaled, do_perm, offsets, E, M_cap, d, n, W1, W2, act, dh,
                   dx_perm, dW1, dW2, err, s, sms, pair_of_row, probs, a_scaled, ds_part,
                   amax_dh, accumulate);
}

int moe_grouped_mlp_bwd_routed_gather(const moe_bf16* x, const moe_bf16* dO, int T, int k,
                                      const moe_bf16* h_saved, const int32_t* pair_of_row,
                                      const float* probs, const int32_t* offsets, int E,
                                      int M_cap, int d, int n, const moe_bf16* W1,
                                      const moe_bf16* W2, int act, int flags, moe_bf16* dh,
                                      moe_bf16* a_scaled, float* ds_part, moe_bf16* dx_perm,
                                      moe_bf16* dW1, moe_bf16* dW2, float* amax_dh, int32_t* err,
                                      void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, d, n);
  if (rc) return rc;
  if (T < 0 || k < 1) return MOE_E_SIZE;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU || (flags & ~MOE_FLAG_ACCUMULATE_DW))
    return MOE_E_ARG;
  const bool accumulate = flags & MOE_FLAG_ACCUMULATE_DW;
  if (!offsets || !W1 || !W2 || !dW1 || !dW2 || !err) return MOE_E_NULL;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M_cap == 0) {
    if (accumulate) return MOE_OK;
    cudaError_t e = cudaMemsetAsync(dW1, 0, static_cast<size_t>(E) * d * n1 * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, static_cast<size_t>(E) * n * d * 2, s);
    return cuda_rc(e);
  }
  if (!x || !dO || !h_saved || !pair_of_row || !probs || !dh || !a_scaled || !ds_part ||
      !dx_perm)
    return MOE_E_NULL;
  if (misaligned(x) || misaligned(dO) || misaligned(h_saved) || misaligned(dh) ||
      misaligned(a_scaled) || misaligned(dx_perm) || misaligned(dW1) || misaligned(dW2) ||
      misaligned(W1) || misaligned(W2))
    return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  // x_perm / dy are not read in gather mode: the token tensors stand in for
  // the map arguments that the gathered operands replace
  return bwd_gemms(x, h_saved, a_scaled, dO, offsets, E, M_cap, d, n, W1, W2, act, dh, dx_perm,
                   dW1, dW2, err, s, sms, pair_of_row, probs, a_scaled, ds_part, amax_dh,
                   accumulate, x, dO, T, k);
}

int moe_router_grad_rows(const float* ds_part, int n_parts, const int32_t* row_of_pair, int T,
                         int k, int M_cap, float* dprobs, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (T < 0 || k < 1 || n_parts < 1 || M_cap < 0) return MOE_E_SIZE;
  if (T == 0) return MOE_OK;
  if (!ds_part || !row_of_pair || !dprobs) return MOE_E_NULL;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_router_grad_rows(ds_part, n_parts, row_of_pair, T * k, M_cap,
                                                     dprobs, sms, s);
  ev_end(s);
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

int moe_mx_quantize_weights(const moe_bf16* W2, int E, int n, int d, const int32_t* offsets,
                            uint8_t* w2_q, uint8_t* w2_s, void* stream) {
  return moe_mx_quantize_weights2(W2, E, n, d, offsets, w2_q, w2_s, nullptr, nullptr, stream);
}

int moe_mx_quantize_weights2(const moe_bf16* W2, int E, int n, int d, const int32_t* offsets,
                             uint8_t* w2_q, uint8_t* w2_s, uint8_t* w2_q_rows,
                             uint8_t* w2_s_rows, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (E < 1 || E > MOE_MAX_EXPERTS || n <= 0 || d <= 0 || n % 128 || d % 128) return MOE_E_SIZE;
  if (!W2 || !w2_q || !w2_s || (w2_q_rows && !w2_s_rows)) return MOE_E_NULL;
  if (misaligned(W2) || misaligned(w2_q) || misaligned(w2_s) || misaligned(w2_q_rows) ||
      misaligned(w2_s_rows))
    return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_mx_quantize_weights(W2, E, n, d, offsets, w2_q, w2_s,
                                                        w2_q_rows, w2_s_rows, sms, s);
  ev_end(s);
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

size_t moe_mx_bwd_workspace_size(int M_cap, int d, int n, int act) {
  if (M_cap < 0 || d <= 0 || n <= 0 || act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU) return 0;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  return carve_mx_bwd(nullptr, M_cap, d, n1, n).bytes;
}

int moe_set_pair_mma(int mode) {
  const int prev = moe::set_pair_mode(mode);
  return prev < 0 ? MOE_E_ARG : prev;
}

size_t moe_mx_bwd_workspace_layout(int M_cap, int d, int n, int act, size_t* offs) {
  if (!offs || M_cap < 0 || d <= 0 || n <= 0 || act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU)
    return 0;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  // a base far from zero, so that every section's address stays positive
  uint8_t* const base = reinterpret_cast<uint8_t*>(static_cast<uintptr_t>(1) << 40);
  const MxBwdWs w = carve_mx_bwd(base, M_cap, d, n1, n);
  const uint8_t* sec[11] = {w.dy_q, w.dy_s, w.dy_qT, w.dy_sT, w.x_qT, w.x_sT,
                            w.a_sT, w.dh_q, w.dh_s, w.dh_qT, w.dh_sT};
  for (int i = 0; i < 11; ++i) offs[i] = static_cast<size_t>(sec[i] - base);
  return w.bytes;
}

size_t moe_workspace_size(int T, int k, int E, int M_cap, int d, int n, int act, int flags) {
  const size_t r = moe_route_workspace_size(T, k, E);
  const size_t m = (flags & MOE_FLAG_MXFP8) ? moe_mx_bwd_workspace_size(M_cap, d, n, act) : 0;
  return r > m ? r : m;
}

int moe_grouped_mlp_fwd_gather(const moe_bf16* x, int T, int k, const int32_t* pair_of_row,
                               const int32_t* offsets, int E, int M_cap, int d, int n,
                               const moe_bf16* W1, const moe_bf16* W2, int act, int flags,
                               moe_bf16* h_saved, moe_bf16* a, moe_bf16* y_perm, float* amax_a,
                               int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, d, n);
  if (rc) return rc;
  if (T < 0 || k < 1) return MOE_E_SIZE;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU || (flags & ~MOE_FLAG_SAVE_H))
    return MOE_E_ARG;
  const bool save_h = flags & MOE_FLAG_SAVE_H;
  if (!offsets || !W1 || !W2 || !err) return MOE_E_NULL;
  if (M_cap == 0) return MOE_OK;
  if (!x || !pair_of_row || !a || !y_perm || (save_h && !h_saved)) return MOE_E_NULL;
  if (misaligned(x) || misaligned(W1) || misaligned(W2) || misaligned(a) || misaligned(y_perm) ||
      (save_h && misaligned(h_saved)))
    return MOE_E_ALIGN;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tw1, ta, tw2;
  if (!map_w(&tw1, W1, E, d, n1, 64) || !map_act(&ta, a, M_cap, n, moe::kBM) ||
      !map_w(&tw2, W2, E, n, d, 64))
    return MOE_E_CUDA;
  moe::GemmArgs g1{};
  g1.offsets = offsets; g1.E = E; g1.M_cap = M_cap; g1.K = d; g1.N = n1; g1.R = 0;
  g1.out = a; g1.ldo = n; g1.out2 = save_h ? h_saved : nullptr; g1.ldo2 = n1; g1.err = err;
  g1.amax = amax_a;
  // A's rows come from x through pair_of_row (copied by the kernel; the A
  // map argument is unused)
  g1.gather_pair = pair_of_row; g1.gather_k = k; g1.gather_T = T;
  g1.gather_src = x; g1.gather_ld = d;
  // H and A leave through staged TMA stores
  CUtensorMap th = tw1, tao;
  if ((save_h && !map_out2(&th, h_saved, M_cap, n1)) || !map_out2(&tao, a, M_cap, n))
    return MOE_E_CUDA;
  g1.tma_out = 1;
  ev_begin(s);
  int launched = 1;
  cudaError_t e = moe::launch_grouped_gemm(moe::GemmKind::kFc1Act, act, tw1, tw1, th, g1, sms, s,
                                           false, &tao, &launched);
  g_split_extra += launched - 1;
  ev_end(s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  moe::GemmArgs g2{};
  g2.offsets = offsets; g2.E = E; g2.M_cap = M_cap; g2.K = n; g2.N = d; g2.R = 0;
  g2.out = y_perm; g2.ldo = d; g2.err = err;
  CUtensorMap ty;
  if (!map_out2(&ty, y_perm, M_cap, d)) return MOE_E_CUDA;
  g2.tma_out = 1;
  e = gemm(moe::GemmKind::kFc2, 0, ta, tw2, ty, g2, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = 2 + g_split_extra;
  return MOE_OK;
}

int moe_grouped_gemm(const moe_bf16* a, const int32_t* offsets, int E, int M_cap, int K, int N,
                     const moe_bf16* B, int b_layout, moe_bf16* out, int32_t* err,
                     void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, K, N);
  if (rc) return rc;
  if (b_layout != MOE_B_KN && b_layout != MOE_B_NK) return MOE_E_ARG;
  if (!offsets || !B || !err) return MOE_E_NULL;
  if (M_cap == 0) return MOE_OK;
  if (!a || !out) return MOE_E_NULL;
  if (misaligned(a) || misaligned(B) || misaligned(out)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the FC2 contraction (B N-major) or the dgrad one (B K-major, rows = N)
  CUtensorMap ta, tb;
  if (!map_act(&ta, a, M_cap, K, moe::kBM)) return MOE_E_CUDA;
  if (b_layout == MOE_B_KN ? !map_w(&tb, B, E, K, N, 64) : !map_w(&tb, B, E, N, K, 128))
    return MOE_E_CUDA;
  moe::GemmArgs g{};
  g.offsets = offsets; g.E = E; g.M_cap = M_cap; g.K = K; g.N = N;
  g.out = out; g.ldo = N; g.err = err;
  CUtensorMap to;
  if (!map_out2(&to, out, M_cap, N)) return MOE_E_CUDA;
  g.tma_out = 1;
  const cudaError_t e = gemm(b_layout == MOE_B_KN ? moe::GemmKind::kFc2 : moe::GemmKind::kDgrad, 0,
                             ta, tb, to, g, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = 1 + g_split_extra;
  return MOE_OK;
}

int moe_activation(const moe_bf16* h, const int32_t* offsets, int E, int M_cap, int n, int act,
                   moe_bf16* a, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, 64, n);
  if (rc) return rc;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU) return MOE_E_ARG;
  if (!offsets) return MOE_E_NULL;
  if (M_cap == 0) return MOE_OK;
  if (!h || !a) return MOE_E_NULL;
  if (misaligned(h) || misaligned(a)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_act_fwd(h, offsets, E, M_cap, n, act, a, sms, s);
  ev_end(s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = 1 + g_split_extra;
  return MOE_OK;
}

int moe_activation_bwd(const moe_bf16* h, const moe_bf16* da, const int32_t* offsets, int E,
                       int M_cap, int n, int act, moe_bf16* dh, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, 64, n);
  if (rc) return rc;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU) return MOE_E_ARG;
  if (!offsets) return MOE_E_NULL;
  if (M_cap == 0) return MOE_OK;
  if (!h || !da || !dh) return MOE_E_NULL;
  if (misaligned(h) || misaligned(da) || misaligned(dh)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_act_bwd(h, da, offsets, E, M_cap, n, act, dh, sms, s);
  ev_end(s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = 1 + g_split_extra;
  return MOE_OK;
}

int moe_mx_quantize_weights_rowwise(const moe_bf16* W, int rows, int cols,
                                    const int32_t* offsets, int E, uint8_t* q, uint8_t* sc,
                                    void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (rows <= 0 || cols <= 0 || rows % 128 || cols % 128) return MOE_E_SIZE;
  if (offsets && (E < 1 || E > MOE_MAX_EXPERTS || rows % E || (rows / E) % 128))
    return MOE_E_SIZE;
  if (!W || !q || !sc) return MOE_E_NULL;
  if (misaligned(W) || misaligned(q)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_mx_quantize_rows_w(W, rows, cols, offsets,
                                                       offsets ? rows / E : rows, q, sc, sms, s);
  ev_end(s);
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

int moe_grouped_mlp_bwd_mx(const moe_bf16* x_perm, const moe_bf16* h_saved,
                           const moe_bf16* dy_perm, const int32_t* offsets, int E, int M_cap,
                           int d, int n, int act, int flags, const moe_mx_bwd* mx,
                           moe_bf16* dh, moe_bf16* dx_perm, moe_bf16* dW1, moe_bf16* dW2,
                           int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  int rc = check_mlp_sizes(E, M_cap, d, n);
  if (rc) return rc;
  if (d % 128 || n % 128 || M_cap % 32) return MOE_E_SIZE;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SRELU ||
      (flags & ~(MOE_FLAG_ACCUMULATE_DW | MOE_FLAG_MX_SEPARATE_DH_QUANT)))
    return MOE_E_ARG;
  const bool accumulate = flags & MOE_FLAG_ACCUMULATE_DW;
  const bool fuse_dh = !(flags & MOE_FLAG_MX_SEPARATE_DH_QUANT);
  if (!offsets || !mx || !dW1 || !dW2 || !err) return MOE_E_NULL;
  const int n1 = (act == MOE_ACT_SRELU) ? n : 2 * n;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M_cap == 0) {
    if (accumulate) return MOE_OK;
    cudaError_t e = cudaMemsetAsync(dW1, 0, static_cast<size_t>(E) * d * n1 * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, static_cast<size_t>(E) * n * d * 2, s);
    return cuda_rc(e);
  }
  if (!x_perm || !h_saved || !dy_perm || !dh || !dx_perm || !mx->a_qT || !mx->a_sT ||
      !mx->w2_q || !mx->w2_s || !mx->w1_q || !mx->w1_s || !mx->workspace ||
      (mx->dx_q && !mx->dx_s))
    return MOE_E_NULL;
  if (misaligned(mx->dx_q)) return MOE_E_ALIGN;
  if (misaligned(x_perm) || misaligned(h_saved) || misaligned(dy_perm) || misaligned(dh) ||
      misaligned(dx_perm) || misaligned(dW1) || misaligned(dW2) || misaligned(mx->a_qT) ||
      misaligned(mx->w2_q) || misaligned(mx->w2_s) || misaligned(mx->w1_q) ||
      misaligned(mx->w1_s) || (reinterpret_cast<uintptr_t>(mx->workspace) & 255u))
    return MOE_E_ALIGN;
  const MxBwdWs ws = carve_mx_bwd(mx->workspace, M_cap, d, n1, n);
  if (mx->ws_bytes < ws.bytes) return MOE_E_WORKSPACE;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;

  CUtensorMap t_dy, t_w2, t_aT, t_dyT, t_dh, t_w1, t_xT, t_dhT, t_dw2, t_dw1;
  if (!map_act(&t_dy, ws.dy_q, M_cap, d, 128, true) ||        // FC2-dgrad A [M, d]
      !map_act(&t_w2, mx->w2_q, E * n, d, 128, true) ||       // FC2-dgrad B [E*n, d]
      !map_act(&t_aT, mx->a_qT, n, M_cap, 128, true) ||       // FC2-wgrad A [n, M]
      !map_act(&t_dyT, ws.dy_qT, d, M_cap, 128, true) ||      // FC2-wgrad B [d, M]
      !map_act(&t_dh, ws.dh_q, M_cap, n1, 128, true) ||       // FC1-dgrad A [M, n1]
      !map_act(&t_w1, mx->w1_q, E * d, n1, 128, true) ||      // FC1-dgrad B [E*d, n1]
      !map_act(&t_xT, ws.x_qT, d, M_cap, 128, true) ||        // FC1-wgrad A [d, M]
      !map_act(&t_dhT, ws.dh_qT, n1, M_cap, 128, true) ||     // FC1-wgrad B [n1, M]
      !map_out3(&t_dw2, dW2, E, n, d, true) || !map_out3(&t_dw1, dW1, E, d, n1, true))
    return MOE_E_CUDA;

  auto quant = [&](const moe_bf16* src, int cols, uint8_t* q, uint8_t* sc, uint8_t* qT,
                   uint8_t* sT) {
    ev_begin(s);
    const cudaError_t e = moe::launch_mx_quantize_act(src, M_cap, cols, offsets, E, q, sc, qT, sT,
                                                      err, true, sms, s);
    ev_end(s);
    return e;
  };
  // 1-3. operands: dY both ways, x transposed, A's transposed scales re-tiled
  cudaError_t e = quant(dy_perm, d, ws.dy_q, ws.dy_s, ws.dy_qT, ws.dy_sT);
  if (e == cudaSuccess) e = quant(x_perm, d, nullptr, nullptr, ws.x_qT, ws.x_sT);
  if (e == cudaSuccess) {
    ev_begin(s);
    e = moe::launch_mx_retile_t(mx->a_sT, M_cap, n, offsets, E, ws.a_sT, sms, s);
    ev_end(s);
  }
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 4. dH = act'(H; dY W2^T); fused: with dH's MXFP8 copies both ways
  moe::MxGemmArgs g{};
  g.offsets = offsets; g.E = E; g.M_cap = M_cap; g.K = d; g.N = n;
  g.a_s = ws.dy_s; g.b_s = mx->w2_s; g.out = dh; g.ldo = n1; g.aux = h_saved; g.ld_aux = n1;
  g.err = err;
  g.a_s_bytes = static_cast<long long>(M_cap) * d / 8;
  g.b_s_bytes = static_cast<long long>(E) * n * d / 32;
  CUtensorMap t_dh_o = t_dy;
  if (fuse_dh) {
    g.dh_q = ws.dh_q; g.dh_s = ws.dh_s; g.dh_qT = ws.dh_qT; g.dh_sT = ws.dh_sT; g.n1 = n1;
    // the fused epilogue stages dH's bf16 blocks and writes them with TMA stores
    if (!map_out2(&t_dh_o, dh, M_cap, n1)) return MOE_E_CUDA;
    g.tma_out = 1;
  }
  e = mx_gemm(moe::MxKind::kDgradAct, act, t_dy, t_w2, t_dh_o, g, sms, s);
  // 5. unfused control: dH both ways in a separate pass
  if (e == cudaSuccess && !fuse_dh) e = quant(dh, n1, ws.dh_q, ws.dh_s, ws.dh_qT, ws.dh_sT);
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 6. dW2_e = A_e^T dY_e
  moe::MxGemmArgs gw2{};
  gw2.offsets = offsets; gw2.E = E; gw2.M_cap = M_cap; gw2.R = n; gw2.N = d;
  gw2.a_s = ws.a_sT; gw2.b_s = ws.dy_sT; gw2.err = err;
  gw2.a_s_bytes = static_cast<long long>(M_cap) * n / 8;
  gw2.b_s_bytes = static_cast<long long>(M_cap) * d / 8;
  gw2.out = dW2; gw2.accumulate = accumulate;
  e = mx_gemm(moe::MxKind::kWgrad, 0, t_aT, t_dyT, t_dw2, gw2, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 7. dX = dH W1^T
  moe::MxGemmArgs gd{};
  gd.offsets = offsets; gd.E = E; gd.M_cap = M_cap; gd.K = n1; gd.N = d;
  gd.a_s = ws.dh_s; gd.b_s = mx->w1_s; gd.out = dx_perm; gd.ldo = d; gd.err = err;
  gd.a_s_bytes = static_cast<long long>(M_cap) * n1 / 8;
  gd.b_s_bytes = static_cast<long long>(E) * d * n1 / 32;
  gd.q_out = mx->dx_q; gd.s_out = mx->dx_q ? mx->dx_s : nullptr;
  CUtensorMap t_dx;
  if (!map_out2(&t_dx, dx_perm, M_cap, d)) return MOE_E_CUDA;
  gd.tma_out = 1;
  e = mx_gemm(moe::MxKind::kDgrad, 0, t_dh, t_w1, t_dx, gd, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  // 8. dW1_e = X_e^T dH_e
  moe::MxGemmArgs gw1{};
  gw1.offsets = offsets; gw1.E = E; gw1.M_cap = M_cap; gw1.R = d; gw1.N = n1;
  gw1.a_s = ws.x_sT; gw1.b_s = ws.dh_sT; gw1.err = err;
  gw1.a_s_bytes = static_cast<long long>(M_cap) * d / 8;
  gw1.b_s_bytes = static_cast<long long>(M_cap) * n1 / 8;
  gw1.out = dW1; gw1.accumulate = accumulate;
  e = mx_gemm(moe::MxKind::kWgrad, 0, t_xT, t_dhT, t_dw1, gw1, sms, s);
  if (e != cudaSuccess) return MOE_E_CUDA;
  g_last_launches = (fuse_dh ? 7 : 8) + g_split_extra;
  return MOE_OK;
}

int moe_mx_quantize(const moe_bf16* src, int rows, int cols, const int32_t* offsets, int E,
                    uint8_t* q, uint8_t* sc, uint8_t* qT, uint8_t* sT, int32_t* err,
                    void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (E < 1 || E > MOE_MAX_EXPERTS || rows < 0 || cols <= 0 || rows % 32 || cols % 32)
    return MOE_E_SIZE;
  if (rows == 0) return MOE_OK;
  if (!src || !offsets || !q || !sc || !err || (qT && !sT)) return MOE_E_NULL;
  if (misaligned(src) || misaligned(q) || misaligned(qT)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_mx_quantize_act(src, rows, cols, offsets, E, q, sc, qT, sT,
                                                    err, false, sms, s);
  ev_end(s);
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

int moe_mx_quantize_tiled(const moe_bf16* src, int rows, int cols, const int32_t* offsets,
                          int E, uint8_t* q, uint8_t* sc, uint8_t* qT, uint8_t* sT,
                          int32_t* err, void* stream) {
  g_last_launches = 0;
  g_split_extra = 0;
  if (E < 1 || E > MOE_MAX_EXPERTS || rows < 0 || cols <= 0 || rows % 32 || cols % 32)
    return MOE_E_SIZE;
  if (rows == 0) return MOE_OK;
  if (cols % 128) return MOE_E_SIZE;
  if (!src || !offsets || !err || (!q && !qT) || (q && !sc) || (qT && !sT)) return MOE_E_NULL;
  if (misaligned(src) || misaligned(q) || misaligned(qT) || misaligned(sc)) return MOE_E_ALIGN;
  const int sms = num_sms_current();
  if (sms <= 0) return MOE_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ev_begin(s);
  const cudaError_t e = moe::launch_mx_quantize_act(src, rows, cols, offsets, E, q, sc, qT, sT,
                                                    err, true, sms, s);
  ev_end(s);
  g_last_launches = 1 + g_split_extra;
  return cuda_rc(e);
}

}  // extern "C"
