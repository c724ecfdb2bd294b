// mx.cu - block-scaled MXFP8 grouped GEMM
// (tcgen05.mma.kind::mxf8f6f4.block_scale) for FC2, the two data gradients
// (FC2's with the dActivation epilogue) and the ragged-K weight gradients;
// the same persistent warp-specialised structure as the bf16 grouped GEMM.
// Its operands come from the quantisers in mx_quant.cu and the FC1
// epilogue.  [TE] "Transformer Engine이 제공하는 세 가지 구성 요소": an MXFP8
// grouped GEMM; [TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩": the
// backward's GroupGemm + dActivation + Quantize/Transpose.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "act.cuh"
#include "gemm.cuh"
#include "mx.cuh"
#include "mxgemm.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- block-scaled GEMM
// Output tiles are 128 x 256, computed as two 128 x 128 block-scaled MMAs per
// 32-element step of K (each half with its own B scale chunk).  A pipeline
// stage holds one 128-byte swizzle atom of K (128 FP8 elements) of A and of
// both B halves plus their three scale chunks: 48 KB of operands for 8.4
// MFLOP, the same bytes-per-FLOP as the bf16 kernel's 128 x 256 x 64 stage
// at twice the tensor rate.
constexpr int QBM = 128, QBN = 256, QHN = 128;   // tile rows, tile columns, MMA N
constexpr int QBK = 128;                          // FP8 elements (= bytes) of K per stage
constexpr int QA_BYTES = QBM * QBK;               // 16 KB
constexpr int QBH_BYTES = QHN * QBK;              // 16 KB per B half
constexpr int QSF_OFF = QA_BYTES + 2 * QBH_BYTES; // scale chunks: SFA, SFB half 0, SFB half 1
constexpr int QSTAGE_BYTES = QSF_OFF + 2048;      // 50 KB (stages stay 1024-byte aligned)
constexpr int QTHREADS = 320;
constexpr int QEPI_WARPS = 8;
constexpr int QTMEM_COLS = 512;
constexpr int QSF_TMEM = QBN;                     // scale columns after the accumulator
constexpr int QSF_COLS = 12;                      // a stage's three chunks, 4 columns each
constexpr int QBOX_BYTES = 32 * 64 * 2;           // staged output box: 32 rows x 64 bf16
// The quantising FC2-dgrad epilogue parks the second half of each
// warpgroup's 128 accumulator columns here (after the scale columns of up
// to six stages, 256..327) so that only 64 of them occupy registers once the
// accumulator is released: columns 384..511
constexpr int QSTASH_TMEM = 384;
// Pair mode (2-SM MMAs, M = 256 over the CTA pair, N = 256): each CTA's
// 32 KB stage holds its 128 rows of A and its 128-column half of B; the
// stage's three scale chunks (its A rows' and both B halves') sit in a
// separate region after the stages, 1.5 KB per stage; all of it is loaded
// by TMA onto the first CTA's full barrier
constexpr int QP_STAGE_BYTES = QA_BYTES + QBH_BYTES;   // 32 KB
constexpr int QP_SF_BYTES = 3 * 512;

// TMEM holds one 256-column accumulator (the scale columns leave no room
// for a second); the epilogue moves it to registers and releases it at once,
// so the next tile's MMAs overlap the conversion and stores.  The weight
// gradient stages its output for TMA stores (one box per epilogue warp plus
// a box of zeros for experts with no rows) and keeps three stages; the other
// kinds keep four.
template <MxKind KIND, bool PAIR = false>
struct QCfg {
  static constexpr bool W = (KIND == MxKind::kWgrad);
  // FC2 and FC1-dgrad store their bf16 output through one staged 32 x 32
  // box (2 KB) per epilogue warp
  static constexpr bool STO = (KIND == MxKind::kFc2 || KIND == MxKind::kDgrad);
  // the quantising FC2-dgrad epilogue transposes dH through one 2 KB box
  // per epilogue warp
  static constexpr bool TBOX = STO || KIND == MxKind::kDgradAct;
  static constexpr int stages = PAIR ? (W ? 5 : 6) : (W ? 3 : 4);
  static constexpr int stage_bytes = PAIR ? QP_STAGE_BYTES : QSTAGE_BYTES;
  // rounded up so that the staging boxes after it stay 1024-byte aligned
  static constexpr int sf_bytes = PAIR ? (stages * QP_SF_BYTES + 1023) / 1024 * 1024 : 0;
  static constexpr int stg_bytes =
      W ? (QEPI_WARPS + 1) * QBOX_BYTES : (TBOX ? QEPI_WARPS * 32 * 32 * 2 : 0);
  // TMEM: accumulator, then each stage's scale columns, then the stash
  static_assert(QSF_TMEM + stages * QSF_COLS <= QSTASH_TMEM &&
                    QSTASH_TMEM + 2 * 64 <= QTMEM_COLS,
                "TMEM columns of the scales and the stash overlap");
};
template <MxKind KIND, bool PAIR = false>
constexpr size_t mx_smem_bytes(int E) {
  using C = QCfg<KIND, PAIR>;
  return 1024 + static_cast<size_t>(C::stages) * C::stage_bytes + C::sf_bytes + C::stg_bytes +
         (2 * C::stages + 4) * 8 + 16 + 2 * (E + 1) * 4;
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
  int e;
  int row0, rows;   // ragged-row kinds: first global row, valid rows
  int m0;           // kWgrad: first output row within the expert
  int n0;           // first accumulator column
  int nh;           // 128-column halves of the tile inside N (1 or 2)
  int kblocks;      // QBK-element reduction steps
  int k0;           // kWgrad: first reduction row (global)
  int klast;        // kWgrad: valid rows of the last step (a multiple of 32)
  bool mc;          // the pair shares (multicasts) this B block
  bool ghost;       // no output: past the expert's row blocks, or past N
};

// Work units of a 2-CTA cluster.  With at least two 128-row blocks, a unit
// is two consecutive row blocks that share one 256-column block of B (CTA r
// takes row block 2i + r; each CTA fetches one 128-column half of B and
// multicasts it into both).  An expert with a single row block pairs along
// N instead: CTA r takes column block 2i + r and loads its own operands.  A
// CTA whose row or column block lies past the expert or past N is a ghost:
// it still fetches and multicasts its half of a shared B block, and still
// frees each stage in both CTAs, but loads, computes and stores nothing
// else.
constexpr int QCL = 2;
constexpr uint16_t kQPair = 0x3;
template <MxKind KIND>
__device__ __forceinline__ int mx_row_blocks(const MxGemmArgs& g, const int* s_off, int e) {
  return (KIND == MxKind::kWgrad) ? g.R / QBM : (s_off[e + 1] - s_off[e] + QBM - 1) / QBM;
}

template <MxKind KIND, bool PAIR = false>
__device__ __forceinline__ int mx_tiles_of_expert(const MxGemmArgs& g, const int* s_off, int e) {
  const int nt = (g.N + QBN - 1) / QBN;
  const int mt = mx_row_blocks<KIND>(g, s_off, e);
  if (!PAIR && mt == 1) return (nt + 1) / 2;
  return ((mt + 1) / 2) * nt;   // pair mode: 256-row units, also for one row block
}

template <MxKind KIND, bool PAIR = false>
__device__ __forceinline__ QTile mx_decode(const MxGemmArgs& g, const int* s_off, const int* s_ts,
                                           int t, int rank) {
  int lo = 0, hi = g.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_ts[mid + 1] <= t) lo = mid + 1;
    else hi = mid;
  }
  const int nt = (g.N + QBN - 1) / QBN;
  const int local = t - s_ts[lo];
  const int mt = mx_row_blocks<KIND>(g, s_off, lo);
  QTile tl;
  tl.e = lo;
  int mi;
  if (!PAIR && mt == 1) {
    tl.mc = false;
    mi = 0;
    tl.n0 = (2 * local + rank) * QBN;
  } else {
    const int pm = local / nt;
    tl.mc = !PAIR;
    mi = 2 * pm + rank;
    tl.n0 = (local - pm * nt) * QBN;
  }
  tl.nh = max(0, min(2, (g.N - tl.n0) / QHN));
  tl.ghost = mi >= mt || tl.nh == 0;
  if constexpr (KIND == MxKind::kWgrad) {
    tl.m0 = mi * QBM;
    tl.k0 = s_off[lo];
    const int kr = s_off[lo + 1] - s_off[lo];
    tl.kblocks = (kr + QBK - 1) / QBK;
    tl.klast = kr - (tl.kblocks - 1) * QBK;
    tl.row0 = 0;
    tl.rows = 0;
  } else {
    tl.row0 = s_off[lo] + mi * QBM;
    tl.rows = tl.ghost ? 0 : min(QBM, s_off[lo + 1] - tl.row0);
    tl.kblocks = g.K / QBK;
    tl.klast = QBK;
    tl.m0 = 0;
    tl.k0 = 0;
  }
  return tl;
}

// 32 fp32 accumulator columns -> 32 bf16 at p (64 bytes)
__device__ __forceinline__ void mx_store_row32(uint16_t* p, const uint32_t (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(p + 8 * k) = make_uint4(
        pack_bf16x2(__uint_as_float(v[8 * k + 0]), __uint_as_float(v[8 * k + 1])),
        pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
        pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
        pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
}

// mx_quant32 from 32 bf16 values packed in pairs (element 2i in the low
// half of p[i]), so that no float copy of the block stays live
__device__ __forceinline__ uint32_t mx_quant32_bf16(const uint32_t (&p)[16], uint32_t (&q)[8]) {
  auto lo16 = [](uint32_t x) { return __uint_as_float(x << 16); };
  auto hi16 = [](uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); };
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(lo16(p[i])), fabsf(hi16(p[i]))));
  const uint32_t code = mx_scale_code(amax);
  const float inv = mx_inv_scale(code);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t lo = e4m3x2(lo16(p[2 * w]) * inv, hi16(p[2 * w]) * inv);
    const uint32_t hi = e4m3x2(lo16(p[2 * w + 1]) * inv, hi16(p[2 * w + 1]) * inv);
    q[w] = lo | (hi << 16);
  }
  return code;
}

// dA columns col..col+31 of one row -> dH (same interleaving as H)
template <int ACT>
__device__ __forceinline__ void mx_dact_row32(const MxGemmArgs& g, long long grow, int col,
                                              const uint32_t (&r)[32]) {
  if constexpr (ACT == MOE_ACT_SRELU) {
    const uint16_t* hp = g.aux + grow * g.ld_aux + col;
    uint16_t* p = g.out + grow * g.ldo + col;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = pack_bf16x2(2.f * fmaxf(bf16_lo(hw[i]), 0.f) * __uint_as_float(r[8 * v + 2 * i]),
                           2.f * fmaxf(bf16_hi(hw[i]), 0.f) * __uint_as_float(r[8 * v + 2 * i + 1]));
      *reinterpret_cast<uint4*>(p + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    const uint16_t* hp = g.aux + grow * g.ld_aux + 2 * col;
    uint16_t* p = g.out + grow * g.ldo + 2 * col;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
      const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};  // (gate, up) pairs
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float gg = bf16_lo(hw[i]), uu = bf16_hi(hw[i]);
        const float da = __uint_as_float(r[4 * v + i]);
        float ph, dph;
        gate_phi_dphi<ACT>(gg, ph, dph);
        o[i] = pack_bf16x2(da * uu * dph, da * ph);
      }
      *reinterpret_cast<uint4*>(p + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// GroupGemm + dActivation + Quantize/Transpose ([TE] "다음 단계: NVFP4, GEMM
// 융합 양자화, A2A 오버랩"; [CuTe] "무엇을 해결하려는가": the low-precision
// output and its transposed copy come from the epilogue, so the bf16
// intermediate is not read again).  One 32-column block of dH for the
// thread's row (16 dA columns when gated, 32 for squared ReLU); the whole
// warp calls it together, its 32 lanes being 32 consecutive rows of one
// expert (a column block of the transposed copy).  Stores the bf16 dH, the
// row-wise codes and scale (row tile of the 128-row tile starting at
// tl_row0) and the transposed codes and scales (K tile of the same rows,
// block q of it).  The transposed copy goes through the warp's 2 KB box in
// shared memory: row r's 16-byte chunk j sits at chunk (j + r/2) % 4 of the
// row, so that both the row writes (8 lanes per 128-byte phase) and the
// column reads (one 64-byte row per load) are free of bank conflicts; lane
// c then quantises column c's 32 values as one block.
template <int ACT>
__device__ __forceinline__ void mx_dact_quant_block(const MxGemmArgs& g, int tl_row0, int q,
                                                    int lane, int hc, const uint32_t* r,
                                                    uint8_t* box, const CUtensorMap* tdh) {
  const int rt = q * 32 + lane;
  const long long grow = static_cast<long long>(tl_row0) + rt;
  const uint16_t* hp = g.aux + grow * g.ld_aux + hc;
  uint32_t pk[16];
  float f[32];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
    const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (ACT == MOE_ACT_SRELU) {
        pk[4 * v + i] = pack_bf16x2(2.f * fmaxf(bf16_lo(hw[i]), 0.f) * __uint_as_float(r[8 * v + 2 * i]),
                                    2.f * fmaxf(bf16_hi(hw[i]), 0.f) * __uint_as_float(r[8 * v + 2 * i + 1]));
      } else {
        const float gg = bf16_lo(hw[i]), uu = bf16_hi(hw[i]);  // (gate, up) pair
        const float da = __uint_as_float(r[4 * v + i]);
        float ph, dph;
        gate_phi_dphi<ACT>(gg, ph, dph);
        pk[4 * v + i] = pack_bf16x2(da * uu * dph, da * ph);
      }
      f[8 * v + 2 * i] = bf16_lo(pk[4 * v + i]);
      f[8 * v + 2 * i + 1] = bf16_hi(pk[4 * v + i]);
    }
  }
  if (tdh == nullptr) {
    uint16_t* p = g.out + grow * g.ldo + hc;
#pragma unroll
    for (int v = 0; v < 4; ++v)
      *reinterpret_cast<uint4*>(p + 8 * v) = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
  }
  // both scale layouts put this 128-row tile's chunk of column group hc / 128 at
  const long long chunk = static_cast<long long>(tl_row0 / 32) * (g.n1 / 128) + hc / 128;
  // row-wise block
  uint32_t qw[8];
  const uint32_t sc = mx_quant32(f, qw);
  uint4* pq = reinterpret_cast<uint4*>(g.dh_q + grow * g.n1 + hc);
  pq[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  pq[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
  g.dh_s[chunk * 512 + mx_chunk_off(rt, (hc >> 5) & 3)] = static_cast<uint8_t>(sc);
  // transposed copy: column hc + c over the warp's 32 rows is one block
  if (tdh != nullptr) {   // the box's previous use was a TMA store: wait until it has read it
    if (lane == 0) bulk_wait_read_0();
    __syncwarp();
  }
  uint8_t* myrow = box + lane * 64;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(myrow + (((j + (lane >> 1)) & 3) * 16)) =
        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
  __syncwarp();
  float col[32];
  const int cj = lane >> 3, ce = (lane & 7) * 2;   // this lane's column: chunk, byte in it
#pragma unroll
  for (int rr = 0; rr < 32; ++rr) {
    const uint16_t b = *reinterpret_cast<const uint16_t*>(
        box + rr * 64 + (((cj + (rr >> 1)) & 3) * 16) + ce);
    col[rr] = __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  __syncwarp();   // the box is free for dH's staged store or the next block
  if (tdh != nullptr) {
    // dH's 32 x 32 block: 64-byte swizzle (chunk j of row r at j ^ ((r/2) % 4)), TMA store
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(myrow + ((j ^ sw) * 16)) =
          make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tdh, box, hc, tl_row0 + q * 32);
      bulk_commit();
    }
  }
  uint32_t cq[8];
  const uint32_t csc = mx_quant32(col, cq);
  uint4* pt = reinterpret_cast<uint4*>(g.dh_qT + static_cast<long long>(hc + lane) * g.M_cap +
                                       (grow - lane));
  pt[0] = make_uint4(cq[0], cq[1], cq[2], cq[3]);
  pt[1] = make_uint4(cq[4], cq[5], cq[6], cq[7]);
  g.dh_sT[chunk * 512 + mx_chunk_off((hc + lane) & 127, q)] = static_cast<uint8_t>(csc);
}

// Persistent warp-specialised block-scaled grouped GEMM in 2-CTA clusters:
// warp 0 TMA producer (operand tiles by tensor maps, B halves multicast
// within the pair, scale chunks by bulk copies), warp 1 TMEM owner and MMA
// issuer (tcgen05.mma ... block_scale; the scale chunks of a stage go to TMEM
// with tcgen05.cp; its commit frees the stage in both CTAs), warps 2-9
// epilogue in two warpgroups, one per 128-column half of the tile.
template <MxKind KIND, int ACT, bool QOUT, bool PAIR>
__global__ void __launch_bounds__(QTHREADS, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmSA,
                   const __grid_constant__ CUtensorMap tmSB, const MxGemmArgs g) {
  constexpr bool W = (KIND == MxKind::kWgrad);
  constexpr bool B_MN = (KIND == MxKind::kFc2);
  // pair mode: one M = 256, N = 256 MMA per 32 of K over both CTAs
  constexpr uint32_t IDESC = PAIR ? idesc_mx(2 * QBM, QBN, false, B_MN) : idesc_mx(QBM, QHN, false, B_MN);
  constexpr int NST = QCfg<KIND, PAIR>::stages;
  constexpr int SBYTES = QCfg<KIND, PAIR>::stage_bytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sf_region = smem + NST * SBYTES;                   // pair mode: scale chunks
  uint8_t* staging = sf_region + QCfg<KIND, PAIR>::sf_bytes;   // one box per epilogue warp
  uint8_t* zero_box = staging + QEPI_WARPS * QBOX_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + QCfg<KIND, PAIR>::stg_bytes);
  uint64_t* empty_bar = full_bar + NST;
  uint64_t* tfull_bar = empty_bar + NST;
  uint64_t* tempty_bar = tfull_bar + 1;
  uint64_t* drain_bar = tempty_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_ts = s_off + (g.E + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int unit0 = blockIdx.x / QCL;     // this cluster's first work unit
  const int unit_step = gridDim.x / QCL;  // clusters in the grid

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full_bar[i], 1);
      // one commit from each CTA's MMA warp; pair mode: the first CTA's
      // commit, multicast to both
      mbar_init(&empty_bar[i], PAIR ? 1 : QCL);
    }
    mbar_init(tfull_bar, 1);
    // pair mode: the first CTA's MMA waits for both CTAs' epilogue warps
    mbar_init(tempty_bar, PAIR ? 2 * QEPI_WARPS : QEPI_WARPS);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (W || (g.tma_out && (QCfg<KIND, PAIR>::STO || KIND == MxKind::kDgradAct))) prefetch_tmap(&tmC);
    if (PAIR) {
      prefetch_tmap(&tmSA);
      prefetch_tmap(&tmSB);
    }
  }
  if (W && warp >= 2) {  // epilogue threads clear the zero box
    for (int i = threadIdx.x - 64; i < QBOX_BYTES / 16; i += 32 * QEPI_WARPS)
      reinterpret_cast<uint4*>(zero_box)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(tmem_slot, QTMEM_COLS);
    else tmem_alloc(tmem_slot, QTMEM_COLS);
  }
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
      const int rows_e = (e < g.E) ? s_off[e + 1] - s_off[e] : 0;
      const bool owned = rows_e >= g.row_min && (g.row_max == 0 || rows_e < g.row_max);
      const int t = (e < g.E && owned) ? mx_tiles_of_expert<KIND, PAIR>(g, s_off, e) : 0;
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
  cluster_sync();  // the peer's barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = s_ts[g.E];

  if (warp == 0 && PAIR) {
    // ---------------------------------------------------------- producer (pair)
    // this CTA's 128 rows of A, its 128-column half of B and three scale
    // chunks; every byte counts on the first CTA's full barrier
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const long long kc_n = g.K / QBK, nq = g.N / QHN, rq = g.R / QBM;
      const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), 0);
      for (int t = unit0; t < total && ok; t += unit_step) {
        const QTile tl = mx_decode<KIND, PAIR>(g, s_off, s_ts, t, rank);
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * SBYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sf_region + stage * QP_SF_BYTES;
          const uint32_t fb = full0 + stage * 8;
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * (QA_BYTES + QBH_BYTES + 3 * 512));
          const int nh = tl.n0 + rank * QHN;   // this CTA's half of B
          long long ca, cb0, cstep;           // scale chunks: A, B half 0, half 1 - half 0
          if constexpr (W) {
            const int kc = tl.k0 + kb * QBK;
            tma_load_2d_pair(sa, &tmA, fb, kc, tl.m0);
            tma_load_2d_pair(sb, &tmB, fb, kc, nh);
            ca = static_cast<long long>(kc / 32) * rq + tl.m0 / QBM;
            cb0 = static_cast<long long>(kc / 32) * nq + tl.n0 / QHN;
            cstep = 1;
          } else {
            tma_load_2d_pair(sa, &tmA, fb, kb * QBK, tl.row0);
            ca = static_cast<long long>(tl.row0 / 32) * kc_n + kb;
            if constexpr (B_MN) {
              tma_load_3d_pair(sb, &tmB, fb, nh, kb * QBK, tl.e);
              cb0 = (static_cast<long long>(tl.e) * kc_n + kb) * nq + tl.n0 / QHN;
              cstep = 1;
            } else {
              tma_load_2d_pair(sb, &tmB, fb, kb * QBK, tl.e * g.N + nh);
              cb0 = ((static_cast<long long>(tl.e) * g.N + tl.n0) / QHN) * kc_n + kb;
              cstep = kc_n;
            }
          }
          // chunks past a buffer read as zeros (rows or columns that are not stored)
          tma_load_2d_pair(ssf, &tmSA, fb, 0, static_cast<int>(2 * ca));
          tma_load_2d_pair(ssf + 512, &tmSB, fb, 0, static_cast<int>(2 * cb0));
          tma_load_2d_pair(ssf + 1024, &tmSB, fb, 0, static_cast<int>(2 * (cb0 + cstep)));
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // give up: the first CTA's full barriers count both CTAs' copies,
        // which this CTA cannot wait on; 1 ms is far longer than a copy takes
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {}
      }
    }
  } else if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool issued[NST];
      uint32_t ipar[NST];
      for (int i = 0; i < NST; ++i) { issued[i] = false; ipar[i] = 0; }
      bool ok = true;
      const long long kc_n = g.K / QBK, nq = g.N / QHN, rq = g.R / QBM;
      for (int t = unit0; t < total && ok; t += unit_step) {
        const QTile tl = mx_decode<KIND, PAIR>(g, s_off, s_ts, t, rank);
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * SBYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sa + QSF_OFF;
          uint64_t* fb = &full_bar[stage];
          // B's halves land in this stage whoever fetched them; A and the
          // scale chunks (small, loaded by each CTA itself) only for a real tile
          mbar_arrive_expect_tx(fb, tl.nh * QBH_BYTES + (tl.ghost ? 0 : QA_BYTES + 512 + tl.nh * 512));
          long long ca, cb0, cstep;  // scale chunks: A, B half 0, B half 1 - half 0
          if constexpr (W) {
            const int kc = tl.k0 + kb * QBK;
            if (!tl.ghost) tma_load_2d(sa, &tmA, fb, kc, tl.m0);
            for (int h = 0; h < tl.nh; ++h) {
              if (tl.mc && h != rank) continue;
              if (tl.mc) tma_load_2d_mc(sb + h * QBH_BYTES, &tmB, fb, kc, tl.n0 + h * QHN, kQPair);
              else tma_load_2d(sb + h * QBH_BYTES, &tmB, fb, kc, tl.n0 + h * QHN);
            }
            ca = static_cast<long long>(kc / 32) * rq + tl.m0 / QBM;
            cb0 = static_cast<long long>(kc / 32) * nq + tl.n0 / QHN;
            cstep = 1;
          } else {
            if (!tl.ghost) tma_load_2d(sa, &tmA, fb, kb * QBK, tl.row0);
            ca = static_cast<long long>(tl.row0 / 32) * kc_n + kb;
            if constexpr (B_MN) {
              for (int h = 0; h < tl.nh; ++h) {
                if (tl.mc && h != rank) continue;
                if (tl.mc)
                  tma_load_3d_mc(sb + h * QBH_BYTES, &tmB, fb, tl.n0 + h * QHN, kb * QBK, tl.e, kQPair);
                else tma_load_3d(sb + h * QBH_BYTES, &tmB, fb, tl.n0 + h * QHN, kb * QBK, tl.e);
              }
              cb0 = (static_cast<long long>(tl.e) * kc_n + kb) * nq + tl.n0 / QHN;
              cstep = 1;
            } else {
              for (int h = 0; h < tl.nh; ++h) {
                if (tl.mc && h != rank) continue;
                const int rb = tl.e * g.N + tl.n0 + h * QHN;
                if (tl.mc) tma_load_2d_mc(sb + h * QBH_BYTES, &tmB, fb, kb * QBK, rb, kQPair);
                else tma_load_2d(sb + h * QBH_BYTES, &tmB, fb, kb * QBK, rb);
              }
              cb0 = ((static_cast<long long>(tl.e) * g.N + tl.n0) / QHN) * kc_n + kb;
              cstep = kc_n;
            }
          }
          if (!tl.ghost) {
            bulk_load(ssf, g.a_s + ca * 512, 512, fb);
            for (int h = 0; h < tl.nh; ++h)
              bulk_load(ssf + 512 * (1 + h), g.b_s + (cb0 + h * cstep) * 512, 512, fb);
          }
          issued[stage] = true;
          ipar[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        for (int i = 0; i < NST; ++i)
          if (issued[i]) {
            const uint32_t a = smem_u32(&full_bar[i]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(a, ipar[i]) && globaltimer_ns() - t0 < kWaitLimitNs) {}
          }
      }
    }
  } else if (warp == 1 && PAIR) {
    // ---------------------------------------------------------- MMA issuer (pair)
    // the first CTA's warp copies both CTAs' scale chunks into their TMEM and
    // issues the M = 256 MMAs; the second CTA's MMA warp has nothing to do
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = unit0; t < total && ok; t += unit_step, ++local) {
        const QTile tl = mx_decode<KIND, PAIR>(g, s_off, s_ts, t, rank);
        if (lane == 0) ok = mbar_wait_cluster(tempty_bar, (local & 1) ^ 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (lane == 0) ok = mbar_wait(&full_bar[stage], phase, abort_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            uint8_t* sa = smem + stage * SBYTES;
            uint8_t* sb = sa + QA_BYTES;
            uint8_t* ssf = sf_region + stage * QP_SF_BYTES;
            const uint32_t sf_t = tmem_base + QSF_TMEM + stage * QSF_COLS;
            // A rows' scales, then both B halves' in consecutive columns
            tmem_cp_sf_pair(sf_t, sdesc_sf(smem_u32(ssf)));
            tmem_cp_sf_pair(sf_t + 4, sdesc_sf(smem_u32(ssf + 512)));
            tmem_cp_sf_pair(sf_t + 8, sdesc_sf(smem_u32(ssf + 1024)));
            const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
            auto mma = [&](int kk) {
              const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(b0 + kk * 4096, QBH_BYTES, 1024)
                                       : sdesc_sw128(b0 + kk * 32, 16, 1024);
              const uint32_t id = IDESC | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
              umma_mx_pair(tmem_base, ad, bd, id, sf_t, sf_t + 4, (kb > 0 || kk > 0) ? 1u : 0u);
            };
            if (W && kb == tl.kblocks - 1 && tl.klast < QBK) {
              // an expert's last reduction step of a weight gradient: one MMA
              // per 32 of its klast rows
              for (int kk = 0; kk < tl.klast / 32; ++kk) mma(kk);
            } else {
#pragma unroll
              for (int kk = 0; kk < QBK / 32; ++kk) mma(kk);
            }
            umma_commit_pair_mc(&empty_bar[stage]);   // frees the stage in both CTAs
          }
          __syncwarp();
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) umma_commit_pair_mc(tfull_bar);   // both CTAs' epilogues
        __syncwarp();
      }
      if (!ok && lane == 0) {
        umma_commit_pair(drain_bar);
        const uint32_t a = smem_u32(drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int t = unit0; t < total && ok; t += unit_step, ++local) {
      const QTile tl = mx_decode<KIND, PAIR>(g, s_off, s_ts, t, rank);
      // the accumulator is free once the epilogue has read the previous tile
      if (lane == 0) ok = mbar_wait(tempty_bar, (local & 1) ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      // One reduction step.  GEN: the generic form (an expert's last step of
      // a weight gradient, which holds klast of its rows, or a tile with one
      // 128-column half inside N); otherwise four K = 32 MMAs per half,
      // unrolled (a runtime MMA count in the same loop body slowed the
      // whole steps' issue).
      auto kstep = [&](int kb, auto gen_c) -> bool {
        constexpr bool GEN = decltype(gen_c)::value;
        if (lane == 0) ok = mbar_wait(&full_bar[stage], phase, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        tc_fence_after();
        if (lane == 0 && !tl.ghost) {
          uint8_t* sa = smem + stage * SBYTES;
          uint8_t* sb = sa + QA_BYTES;
          uint8_t* ssf = sa + QSF_OFF;
          const uint32_t sf_t = tmem_base + QSF_TMEM + stage * QSF_COLS;
          tmem_cp_sf(sf_t, sdesc_sf(smem_u32(ssf)));
          const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
          auto mma = [&](int kk, int h) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint32_t id = IDESC | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4);
            const uint32_t bh = b0 + h * QBH_BYTES;
            const uint64_t bd = B_MN ? sdesc_sw128(bh + kk * 4096, QBH_BYTES, 1024)
                                     : sdesc_sw128(bh + kk * 32, 16, 1024);
            umma_mx(tmem_base + h * QHN, ad, bd, id, sf_t, sf_t + 4 * (1 + h),
                    (kb > 0 || kk > 0) ? 1u : 0u);
          };
          if constexpr (GEN) {
            for (int h = 0; h < tl.nh; ++h)
              tmem_cp_sf(sf_t + 4 * (1 + h), sdesc_sf(smem_u32(ssf + 512 * (1 + h))));
            // an expert's last reduction step of a weight gradient holds
            // klast (a multiple of 32) of its rows: one MMA per 32 of them
            const int kk_n = (W && kb == tl.kblocks - 1) ? tl.klast / 32 : QBK / 32;
            for (int kk = 0; kk < kk_n; ++kk)
              for (int h = 0; h < tl.nh; ++h) mma(kk, h);
          } else {
            tmem_cp_sf(sf_t + 4, sdesc_sf(smem_u32(ssf + 512)));
            tmem_cp_sf(sf_t + 8, sdesc_sf(smem_u32(ssf + 1024)));
#pragma unroll
            for (int kk = 0; kk < QBK / 32; ++kk) {
              mma(kk, 0);
              mma(kk, 1);
            }
          }
        }
        // the stage is free in both CTAs once both MMA warps have read it
        if (lane == 0) umma_commit_mc(&empty_bar[stage], kQPair);
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1; }
        return true;
      };
      const bool short_last = W && tl.kblocks > 0 && tl.klast < QBK;
      const int whole = short_last ? tl.kblocks - 1 : tl.kblocks;
      if (tl.nh == 2) {
        for (int kb = 0; kb < whole; ++kb)
          if (!kstep(kb, BoolC<false>{})) break;
      } else {
        for (int kb = 0; kb < whole; ++kb)
          if (!kstep(kb, BoolC<true>{})) break;
      }
      if (ok && short_last) kstep(tl.kblocks - 1, BoolC<true>{});
      if (!ok) break;
      if (lane == 0) umma_commit(tfull_bar);
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
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quadrant
    const int wg = (warp - 2) >> 2;      // 128-column half of the tile
    const int r = q * 32 + lane;
    uint8_t* my_box = staging + (warp - 2) * QBOX_BYTES;
    // pair mode: the first CTA's MMA warp waits for this CTA's epilogue too
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(tempty_bar), 0) : 0u;
    auto release = [&]() {
      if (PAIR && rank != 0) mbar_arrive_cluster(tempty0);
      else mbar_arrive(tempty_bar);
    };
    int local = 0;
    for (int t = unit0; t < total; t += unit_step, ++local) {
      const QTile tl = mx_decode<KIND, PAIR>(g, s_off, s_ts, t, rank);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(tfull_bar, local & 1, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const bool zero = W && tl.kblocks == 0;
      // accumulating weight gradients leave an empty expert's untouched
      const bool mine = wg < tl.nh && !tl.ghost && !(zero && g.accumulate);
      if constexpr (KIND == MxKind::kDgradAct && QOUT) {
        // GroupGemm + dActivation + Quantize/Transpose: columns 64..127 of
        // the warpgroup's half go to the TMEM stash, 0..63 to registers;
        // then the accumulator is released and the dH blocks are produced
        const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tb = tmem_base + lanes + wg * QHN;
        const uint32_t st = tmem_base + lanes + QSTASH_TMEM + wg * 64;
        uint32_t v0[32], v1[32];
        if (mine) {
          tmem_ld32(tb + 64, v0);
          tmem_wait_ld();
          tmem_st32(st, v0);
          tmem_ld32(tb + 96, v0);
          tmem_wait_ld();
          tmem_st32(st + 32, v0);
          tmem_ld32(tb, v0);
          tmem_ld32(tb + 32, v1);
          tmem_wait_ld();
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release();
        // offsets are multiples of 32: a warp's 32 rows are all valid or none
        if (!mine || q * 32 >= tl.rows) continue;
        constexpr int BLK = (ACT == MOE_ACT_SRELU) ? 32 : 16;   // dA columns per dH block
        const int col0 = tl.n0 + wg * QHN;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          if (c == 2) {
            tmem_ld32(st, v0);
            tmem_ld32(st + 32, v1);
            tmem_wait_ld();
          }
          const uint32_t* src = (c & 1) ? v1 : v0;
#pragma unroll
          for (int b = 0; b < 32 / BLK; ++b) {
            const int dcol = col0 + 32 * c + b * BLK;          // first dA column
            mx_dact_quant_block<ACT>(g, tl.row0, q, lane, (ACT == MOE_ACT_SRELU) ? dcol : 2 * dcol,
                                     src + b * BLK, staging + (warp - 2) * (32 * 32 * 2),
                                     g.tma_out ? &tmC : nullptr);
          }
        }
        continue;
      }
      if constexpr (QOUT && KIND != MxKind::kDgradAct) {
        // GroupGemm + Quantize ([TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A
        // 오버랩"): the bf16 output and its row-wise MXFP8 copy.  The
        // accumulator is read one 32-column chunk at a time and rounded to
        // bf16 at once (half the registers of the fp32 values), then
        // released.  Each chunk leaves as a staged TMA store of the bf16
        // values (64-byte swizzle, as below) and, from the thread that owns
        // the row, its 32 E4M3 codes quantised from those bf16 values; the
        // four E8M0 scales of the thread's 128 columns leave as one word.
        uint32_t pk4[4][16];
        if (mine) {
          const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + wg * QHN;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t t32[32];
            tmem_ld32(tb + c * 32, t32);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk4[c][i] = pack_bf16x2(__uint_as_float(t32[2 * i]), __uint_as_float(t32[2 * i + 1]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release();
        // offsets are multiples of 32: a warp's 32 rows are all valid or none
        if (!mine || q * 32 >= tl.rows) continue;
        const int col0 = tl.n0 + wg * QHN;
        const long long grow = tl.row0 + r;
        const bool staged = g.tma_out && q * 32 + 32 <= tl.rows;
        uint8_t* box = staging + (warp - 2) * (32 * 32 * 2);
        uint32_t s4 = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (staged) {
            if (lane == 0) bulk_wait_read_0();     // the box's previous store has read it
            __syncwarp();
            uint8_t* row = box + lane * 64;
            const int sw = (lane >> 1) & 3;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) =
                  make_uint4(pk4[c][4 * j], pk4[c][4 * j + 1], pk4[c][4 * j + 2], pk4[c][4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, box, col0 + c * 32, tl.row0 + q * 32);
              bulk_commit();
            }
          } else {
            uint4* p = reinterpret_cast<uint4*>(g.out + grow * g.ldo + col0 + c * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              p[k] = make_uint4(pk4[c][4 * k], pk4[c][4 * k + 1], pk4[c][4 * k + 2], pk4[c][4 * k + 3]);
          }
          uint32_t qw[8];
          s4 |= mx_quant32_bf16(pk4[c], qw) << (8 * c);
          uint4* pq = reinterpret_cast<uint4*>(g.q_out + grow * g.N + col0 + c * 32);
          pq[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
          pq[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
        }
        // N and col0 are multiples of 128: the word is 4-byte aligned when
        // the scale buffer is
        uint8_t* sp = g.s_out + grow * (g.N / 32) + col0 / 32;
        if ((reinterpret_cast<uintptr_t>(sp) & 3) == 0) {
          *reinterpret_cast<uint32_t*>(sp) = s4;
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) sp[c] = static_cast<uint8_t>(s4 >> (8 * c));
        }
        continue;
      }
      uint32_t v[4][32];
      if (mine && !zero) {
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + wg * QHN;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tb + c * 32, v[c]);
        tmem_wait_ld();
      }
      // release the accumulator: the next tile's MMAs may start
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release();
      if (!mine) continue;
      const int col0 = tl.n0 + wg * QHN;
      if constexpr (W) {
        if (g.accumulate && !zero) {
          const uint16_t* op = g.out + (static_cast<long long>(tl.e) * g.R + tl.m0 + q * 32 + lane) * g.N + col0;
#pragma unroll
          for (int c = 0; c < 4; ++c) add_bf16_row32(op + 32 * c, v[c]);
        }
        if (zero) {
          // expert with no rows: its weight gradient is zero
          if (lane == 0) {
            tma_store_3d(&tmC, zero_box, col0, tl.m0 + q * 32, tl.e);
            tma_store_3d(&tmC, zero_box, col0 + 64, tl.m0 + q * 32, tl.e);
            bulk_commit();
          }
          __syncwarp();
        } else {
          // stage each 32-row x 64-column box (128-byte swizzle: 16-byte
          // chunk j of row r at j ^ (r % 8)) and write it with a TMA store
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (lane == 0) bulk_wait_read_0();     // the box's previous store has read it
            __syncwarp();
            uint8_t* row = my_box + lane * 128;
            const int sw = lane & 7;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t (&src)[32] = v[2 * h + (j >> 2)];
              const int b = 8 * (j & 3);
              *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) = make_uint4(
                  pack_bf16x2(__uint_as_float(src[b + 0]), __uint_as_float(src[b + 1])),
                  pack_bf16x2(__uint_as_float(src[b + 2]), __uint_as_float(src[b + 3])),
                  pack_bf16x2(__uint_as_float(src[b + 4]), __uint_as_float(src[b + 5])),
                  pack_bf16x2(__uint_as_float(src[b + 6]), __uint_as_float(src[b + 7])));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmC, my_box, col0 + h * 64, tl.m0 + q * 32, tl.e);
              bulk_commit();
            }
          }
        }
      } else if (QCfg<KIND, PAIR>::STO && g.tma_out && q * 32 + 32 <= tl.rows) {
        // the warp's 32 rows all lie in the expert: stage each 32 x 32 chunk
        // (64-byte swizzle: 16-byte chunk j of row r at j ^ ((r / 2) % 4))
        // and write it with a TMA store
        uint8_t* box = staging + (warp - 2) * (32 * 32 * 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (lane == 0) bulk_wait_read_0();       // the box's previous store has read it
          __syncwarp();
          uint8_t* row = box + lane * 64;
          const int sw = (lane >> 1) & 3;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) = make_uint4(
                pack_bf16x2(__uint_as_float(v[c][8 * j + 0]), __uint_as_float(v[c][8 * j + 1])),
                pack_bf16x2(__uint_as_float(v[c][8 * j + 2]), __uint_as_float(v[c][8 * j + 3])),
                pack_bf16x2(__uint_as_float(v[c][8 * j + 4]), __uint_as_float(v[c][8 * j + 5])),
                pack_bf16x2(__uint_as_float(v[c][8 * j + 6]), __uint_as_float(v[c][8 * j + 7])));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, box, col0 + c * 32, tl.row0 + q * 32);
            bulk_commit();
          }
        }
      } else {
        if (r < tl.rows) {
          const long long grow = tl.row0 + r;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if constexpr (KIND == MxKind::kDgradAct) mx_dact_row32<ACT>(g, grow, col0 + c * 32, v[c]);
            else mx_store_row32(g.out + grow * g.ldo + col0 + c * 32, v[c]);
          }
        }
      }
    }
    if ((W || QCfg<KIND, PAIR>::TBOX) && lane == 0) bulk_wait_all();  // staged stores done before the CTA exits
    __syncwarp();
  }
  tc_fence_before();
  // no CTA leaves while its peer may still multicast into it or arrive on it
  cluster_sync();
  if (*abort_flag && threadIdx.x == 0) set_err(g.err, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, QTMEM_COLS);
    else tmem_dealloc(tmem_base, QTMEM_COLS);
  }
}

// 2-D u8 map over a scale buffer seen as rows of 256 bytes; a box of two
// rows is one 512-byte chunk (pair mode loads the chunks with TMA)
PFN_cuTensorMapEncodeTiled_v12000 mx_encode_fn() {
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
bool map_scale_chunks(CUtensorMap* m, const uint8_t* base, long long bytes) {
  auto fn = mx_encode_fn();
  if (!fn || base == nullptr || bytes < 512 || bytes % 256) return false;
  cuuint64_t gdim[2] = {256, static_cast<cuuint64_t>(bytes / 256)};
  cuuint64_t gstride[1] = {256};
  cuuint32_t bdim[2] = {256, 2}, estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), gdim, gstride, bdim,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <MxKind KIND, int ACT, bool QOUT = false, bool PAIR = false>
cudaError_t launch_mx_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const MxGemmArgs& g, int num_sms, cudaStream_t st) {
  auto kern = mx_gemm_kernel<KIND, ACT, QOUT, PAIR>;
  static_assert(mx_smem_bytes<KIND, PAIR>(MOE_MAX_EXPERTS) <= 227 * 1024,
                "dynamic shared memory above the 227 KB a CTA may have");
  const size_t smem = mx_smem_bytes<KIND, PAIR>(MOE_MAX_EXPERTS);
  CUtensorMap tsa = ta, tsb = ta;   // any valid maps when not in pair mode
  if (PAIR && (!map_scale_chunks(&tsa, g.a_s, g.a_s_bytes) ||
               !map_scale_chunks(&tsb, g.b_s, g.b_s_bytes)))
    return cudaErrorInvalidValue;
  // grid size and shared-memory attribute, set up once per device and
  // instantiation
  static int grid_of[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = QCL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(QTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int& grid = grid_of[dev];
  if (grid == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    const int most = num_sms / QCL;
    grid = QCL * ((clusters > 0 && clusters < most) ? clusters : most);
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tsa, tsb, g);
}

// pair mode for this launch (moe_set_pair_mma), only with the scale buffers'
// sizes known.  Automatic: always for the ragged-row kinds, whose 34 KB
// stages beat the single-CTA tiles' 50 KB even on a layer of one-row-block
// experts (Zipf MXFP8 training layer, 128 rows per expert on average: FC2
// 1.03 -> 0.86 ms, FC2-dgrad 1.01 -> 0.85, FC1-dgrad 1.84 -> 1.45); the
// weight gradients from 256 rows per expert on average, as the bf16 GEMM
// (on that layer they measured 1.84 / 3.64 ms single against 1.87 / 3.71).
bool mx_use_pair(MxKind kind, const MxGemmArgs& g) {
  if (g.a_s_bytes <= 0 || g.b_s_bytes <= 0) return false;
  const int m = pair_mode();
  if (m == kPairNever) return false;
  if (m == kPairAlways || kind != MxKind::kWgrad) return true;
  return static_cast<long long>(g.M_cap) >= static_cast<long long>(kPairRows) * g.E;
}

template <MxKind KIND, int ACT, bool QOUT = false>
cudaError_t launch_mx(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                      const MxGemmArgs& g, int num_sms, cudaStream_t st) {
  return mx_use_pair(KIND, g) ? launch_mx_t<KIND, ACT, QOUT, true>(ta, tb, tc, g, num_sms, st)
                              : launch_mx_t<KIND, ACT, QOUT, false>(ta, tb, tc, g, num_sms, st);
}

}  // namespace

cudaError_t launch_mx_gemm(MxKind kind, int act, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const MxGemmArgs& g, int num_sms,
                           cudaStream_t st, int* launched) {
  if (launched) *launched = 1;
  if (kind == MxKind::kWgrad && g.row_min == 0 && g.row_max == 0 && g.E > 1 &&
      pair_mode() == kPairAuto && g.a_s_bytes > 0 && g.b_s_bytes > 0 &&
      !mx_use_pair(kind, g)) {
    // hot experts (kPairRows reduction rows or more) with 2-SM tiles, then
    // the rest single-CTA; the two launches write disjoint experts, experts
    // with no rows belong to the second
    MxGemmArgs gh = g;
    gh.row_min = kPairRows;
    MxGemmArgs gl = g;
    gl.row_max = kPairRows;
    cudaError_t e = launch_mx_t<MxKind::kWgrad, 0, false, true>(ta, tb, tc, gh, num_sms, st);
    if (e != cudaSuccess) return e;
    if (launched) *launched = 2;
    return launch_mx_t<MxKind::kWgrad, 0, false, false>(ta, tb, tc, gl, num_sms, st);
  }
  switch (kind) {
    // the quantising epilogue (GroupGemm + Quantize) is its own instantiation,
    // so that the plain one keeps its registers
    case MxKind::kFc2:
      return g.q_out ? launch_mx<MxKind::kFc2, 0, true>(ta, tb, tc, g, num_sms, st)
                     : launch_mx<MxKind::kFc2, 0>(ta, tb, tc, g, num_sms, st);
    case MxKind::kDgrad:
      return g.q_out ? launch_mx<MxKind::kDgrad, 0, true>(ta, tb, tc, g, num_sms, st)
                     : launch_mx<MxKind::kDgrad, 0>(ta, tb, tc, g, num_sms, st);
    case MxKind::kWgrad: return launch_mx<MxKind::kWgrad, 0>(ta, tb, tc, g, num_sms, st);
    case MxKind::kDgradAct:
      if (g.dh_q != nullptr) {
        // GroupGemm + dActivation + Quantize/Transpose
        if (!g.dh_s || !g.dh_qT || !g.dh_sT || g.n1 <= 0 || g.n1 % 128) return cudaErrorInvalidValue;
        switch (act) {
          case MOE_ACT_SWIGLU: return launch_mx<MxKind::kDgradAct, MOE_ACT_SWIGLU, true>(ta, tb, tc, g, num_sms, st);
          case MOE_ACT_GEGLU: return launch_mx<MxKind::kDgradAct, MOE_ACT_GEGLU, true>(ta, tb, tc, g, num_sms, st);
          case MOE_ACT_SRELU: return launch_mx<MxKind::kDgradAct, MOE_ACT_SRELU, true>(ta, tb, tc, g, num_sms, st);
          default: return cudaErrorInvalidValue;
        }
      }
      switch (act) {
        case MOE_ACT_SWIGLU: return launch_mx<MxKind::kDgradAct, MOE_ACT_SWIGLU>(ta, tb, tc, g, num_sms, st);
        case MOE_ACT_GEGLU: return launch_mx<MxKind::kDgradAct, MOE_ACT_GEGLU>(ta, tb, tc, g, num_sms, st);
        case MOE_ACT_SRELU: return launch_mx<MxKind::kDgradAct, MOE_ACT_SRELU>(ta, tb, tc, g, num_sms, st);
        default: return cudaErrorInvalidValue;
      }
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
