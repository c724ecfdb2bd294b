// mx.cu - MXFP8 kernels:
//   * mx_quantize_weights: W2 [E, n, d] bf16 -> E4M3 codes [E, n, d] and
//     E8M0 scales over 32 consecutive rows (FC2's reduction index) per
//     column, in the MMA-tiled layout (see mx.cuh).
//   * mx_quantize_act: group-aware quantiser of a ragged [rows, cols]
//     activation: row-wise 1x32 blocks, plus the transposed copy with
//     column-wise 32x1 blocks that never cross an expert's rows.
//   * mx_fc2: block-scaled MXFP8 grouped GEMM Y_e = A_e W2_e
//     (tcgen05.mma.kind::mxf8f6f4.block_scale), same persistent
//     warp-specialised structure as the bf16 grouped GEMM.
// [CuTe] "무엇을 해결하려는가" and "핵심 아이디어": MXFP8 output and transposed
// output; [TE] "Transformer Engine이 제공하는 세 가지 구성 요소": group-aware
// MXFP8 quantisation and an MXFP8 grouped GEMM.
#include <cuda_runtime.h>

#include "mx.cuh"
#include "mxgemm.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- weights
// one thread: 8 consecutive columns x one 32-row block of one expert
__global__ void __launch_bounds__(256)
    mx_quantize_weights_kernel(const uint4* __restrict__ w, int E, int n, int d,
                               uint2* __restrict__ q, uint8_t* __restrict__ s) {
  const int d8 = d / 8;
  const long long total = static_cast<long long>(E) * (n / 32) * d8;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(g % d8);
    const long long eb = g / d8;
    const int b = static_cast<int>(eb % (n / 32));
    const int e = static_cast<int>(eb / (n / 32));
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

// ---------------------------------------------------------------- activations
// one warp: a 32-row block (inside one expert) x a 32-column block
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
    uint32_t qw[8];
    const uint32_t sc = mx_quant32(v, qw);
    uint4* qo = reinterpret_cast<uint4*>(q + static_cast<long long>(r) * cols + cb * 32);
    qo[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    qo[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    s[static_cast<long long>(r) * cb_n + cb] = static_cast<uint8_t>(sc);
    if (qT) {
      uint32_t my_sc = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        uint32_t code;
        const uint32_t scj = mx_quant_lanes(v[j], code);
        qT[static_cast<long long>(cb * 32 + j) * rows + r] = static_cast<uint8_t>(code);
        if (lane == j) my_sc = scj;
      }
      sT[static_cast<long long>(cb * 32 + lane) * (rows / 32) + rb] = static_cast<uint8_t>(my_sc);
    }
  }
}

// ---------------------------------------------------------------- block-scaled FC2
constexpr int QBM = 128, QBN = 128, QBK = 128;  // QBK: FP8 elements (= bytes) of K
constexpr int QSTAGES = 6;
constexpr int QA_BYTES = QBM * QBK;               // 16 KB
constexpr int QB_BYTES = QBN * QBK;               // 16 KB
constexpr int QSTAGE_BYTES = QA_BYTES + QB_BYTES + 1024;  // + SFA, SFB chunks
constexpr int QTHREADS = 192;
constexpr int QTMEM_COLS = 512;
constexpr int QSF_TMEM = 2 * QBN;                 // scale columns after the accumulators

constexpr size_t mx_smem_bytes(int E) {
  return 1024 + static_cast<size_t>(QSTAGES) * QSTAGE_BYTES + (2 * QSTAGES + 5) * 8 + 16 +
         2 * (E + 1) * 4;
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: A/B E4M3 (format 0),
// bit 15/16 A/B major, bits 17-22 N>>3, bit 23 scale type (1 = E8M0),
// bits 24-28 M>>4; scale-factor byte selectors: B bits 4-5, A bits 29-30.
constexpr uint32_t idesc_mx(int M, int N, bool a_mn, bool b_mn) {
  return ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// no-swizzle descriptor of a 512-byte scale chunk (32 rows x 16 bytes,
// 8-row core matrices 128 bytes apart)
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(512 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

struct QTile {
  int e, row0, rows, n0;
};

__global__ void __launch_bounds__(QTHREADS, 1)
    mx_fc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const MxFc2Args g) {
  constexpr uint32_t IDESC = idesc_mx(QBM, QBN, false, true);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + QSTAGES * QSTAGE_BYTES);
  uint64_t* empty_bar = full_bar + QSTAGES;
  uint64_t* tfull_bar = empty_bar + QSTAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_ts = s_off + (g.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = g.d / QBN;
  const int kblocks = g.n / QBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < QSTAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, QTMEM_COLS);
  if (warp == 2) {
    // offsets: non-decreasing multiples of 32 within [0, M_cap]
    bool bad = false;
    for (int i = lane; i <= g.E; i += 32) {
      const int v = g.offsets[i];
      if (v < 0 || v > g.M_cap || (v & 31)) bad = true;
      s_off[i] = min(max(v, 0), g.M_cap) & ~31;
    }
    __syncwarp();
    if (lane == 0) {
      int prev = 0;
      for (int i = 0; i <= g.E; ++i) {
        if (s_off[i] < prev) { bad = true; s_off[i] = prev; }
        prev = s_off[i];
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) set_err(g.err, MOE_DEV_BAD_OFFSETS);
    __syncwarp();
    int carry = 0;
    for (int base = 0; base < g.E; base += 32) {
      const int e = base + lane;
      const int t = (e < g.E) ? ((s_off[e + 1] - s_off[e] + QBM - 1) / QBM) * nt : 0;
      int v = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (e < g.E) s_ts[e] = carry + v - t;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_ts[g.E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_ts[g.E];

  auto decode = [&](int t) {
    int lo = 0, hi = g.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_ts[mid + 1] <= t) lo = mid + 1;
      else hi = mid;
    }
    QTile tl;
    tl.e = lo;
    const int local = t - s_ts[lo];
    const int mi = local / nt;
    tl.n0 = (local - mi * nt) * QBN;
    tl.row0 = s_off[lo] + mi * QBM;
    tl.rows = min(QBM, s_off[lo + 1] - tl.row0);
    return tl;
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool issued[QSTAGES];
      uint32_t ipar[QSTAGES];
      for (int i = 0; i < QSTAGES; ++i) { issued[i] = false; ipar[i] = 0; }
      bool ok = true;
      const long long sa_stride = g.n / 128;       // chunks per 32-row group of A scales
      const long long sw_expert = static_cast<long long>(g.n / 32) * g.d;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const QTile tl = decode(t);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * QSTAGE_BYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sb + QB_BYTES;
          uint64_t* fb = &full_bar[stage];
          mbar_arrive_expect_tx(fb, QSTAGE_BYTES);
          tma_load_2d(sa, &tmA, fb, kb * QBK, tl.row0);
          tma_load_3d(sb, &tmB, fb, tl.n0, kb * QBK, tl.e);
          bulk_load(ssf, g.a_s + ((tl.row0 / 32) * sa_stride + kb) * 512, 512, fb);
          bulk_load(ssf + 512,
                    g.w2_s + tl.e * sw_expert + (static_cast<long long>(kb) * (g.d / 128) + tl.n0 / 128) * 512,
                    512, fb);
          issued[stage] = true;
          ipar[stage] = phase;
          if (++stage == QSTAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        for (int i = 0; i < QSTAGES; ++i)
          if (issued[i]) {
            const uint32_t a = smem_u32(&full_bar[i]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(a, ipar[i]) && globaltimer_ns() - t0 < kWaitLimitNs) {}
          }
      }
    }
  } else if (warp == 1) {
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      if (lane == 0) ok = mbar_wait(&tempty_bar[buf], aph ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * QBN;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (lane == 0) ok = mbar_wait(&full_bar[stage], phase, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          uint8_t* sa = smem + stage * QSTAGE_BYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sb + QB_BYTES;
          const uint32_t sfa_t = tmem_base + QSF_TMEM + stage * 8;
          const uint32_t sfb_t = sfa_t + 4;
          tmem_cp_sf(sfa_t, sdesc_sf(smem_u32(ssf)));
          tmem_cp_sf(sfb_t, sdesc_sf(smem_u32(ssf + 512)));
          const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
#pragma unroll
          for (int kk = 0; kk < QBK / 32; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b0 + kk * 4096, QB_BYTES, 1024);
            const uint32_t id = IDESC | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
            umma_mx(d_tmem, ad, bd, id, sfa_t, sfb_t, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[stage]);
        }
        __syncwarp();
        if (++stage == QSTAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&tfull_bar[buf]);
      __syncwarp();
    }
    if (!ok && lane == 0) {
      umma_commit(drain_bar);
      const uint32_t a = smem_u32(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      const QTile tl = decode(t);
      const int buf = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&tfull_bar[buf], aph, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * QBN;
#pragma unroll 1
      for (int c = 0; c < QBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tb + c * 32, v);
        tmem_wait_ld();
        if (r < tl.rows) {
          uint16_t* p = g.out + static_cast<long long>(tl.row0 + r) * g.d + tl.n0 + c * 32;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(p + 8 * k) = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * k + 0]), __uint_as_float(v[8 * k + 1])),
                pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) set_err(g.err, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, QTMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_mx_quantize_weights(const uint16_t* w2, int E, int n, int d, uint8_t* q,
                                       uint8_t* s, int num_sms, cudaStream_t st) {
  const long long threads = static_cast<long long>(E) * (n / 32) * (d / 8);
  const long long want = (threads + 255) / 256;
  const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
  mx_quantize_weights_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(w2), E, n, d, reinterpret_cast<uint2*>(q), s);
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_act(const uint16_t* src, int rows, int cols, const int32_t* offsets,
                                   int E, uint8_t* q, uint8_t* s, uint8_t* qT, uint8_t* sT,
                                   int32_t* err, int num_sms, cudaStream_t st) {
  const long long warps = static_cast<long long>(rows / 32) * (cols / 32);
  const long long want = (warps * 32 + 255) / 256;
  const int blocks = static_cast<int>(want < 16LL * num_sms ? want : 16LL * num_sms);
  mx_quantize_act_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(
      reinterpret_cast<const uint4*>(src), rows, cols, offsets, E, q, s, qT, sT, err);
  return cudaGetLastError();
}

cudaError_t launch_mx_fc2(const CUtensorMap& ta, const CUtensorMap& tb, const MxFc2Args& g,
                          int num_sms, cudaStream_t st) {
  const size_t smem = mx_smem_bytes(MOE_MAX_EXPERTS);
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(mx_fc2_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  mx_fc2_kernel<<<num_sms, QTHREADS, smem, st>>>(ta, tb, g);
  return cudaGetLastError();
}

}  // namespace moe
