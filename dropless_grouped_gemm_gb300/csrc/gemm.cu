// gemm.cu - persistent grouped GEMM over ragged expert groups (sm_103a).
//
// One kernel template covers the six contractions of the expert MLP:
//   FC1 + activation, FC2, FC2-dgrad + dActivation, FC1-dgrad (ragged rows)
//   and the two weight gradients (ragged reduction).
// [TE] "최적화 1: grouped GEMM": one launch over all experts with their real
// row counts; counts/offsets are read on the device, so nothing is copied to
// the host.  [CuTe] "핵심 아이디어": the GLU is applied in the epilogue.
// [Sonic] "IO 숨기기" / "GEMM Overlapping": warp specialisation (producer,
// MMA, epilogue) and software pipelining hide the epilogue's IO.
//
// Roles (320 threads, one CTA per SM, persistent over a static tile order):
//   warp 0     TMA producer (one lane): 4-stage ring of 48 KB stages
//   warp 1     TMEM owner + MMA issuer (one lane): tcgen05.mma 128x256x16
//   warps 2-9  epilogue, two warpgroups splitting the tile's columns:
//              tcgen05.ld (warp w reads TMEM lanes 32*(w%4)..), activation /
//              derivative math, stores to global
// Two 256-column fp32 accumulators in TMEM let tile i+1's MMAs overlap
// tile i's epilogue.
//
// Pair mode (the ragged-row kinds on experts of 256 rows or more): the two
// CTAs of a cluster compute a 256 x 256 tile with 2-SM MMAs
// (tcgen05.mma.cta_group::2, issued by the first CTA): each CTA loads its
// own 128 rows of A and one 128-column half of B into 32 KB stages, six of
// them, and holds its 128 rows of the accumulator in its own TMEM.
#include <cuda_runtime.h>

#include <atomic>

#include "act.cuh"
#include "gemm.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = kBM, BN = kBN, BK = kBK, UK = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MN_BOX_BYTES = 64 * BK * 2;  // one 64(MN) x 64(K) box: 8 KB
constexpr int NUM_THREADS = 320;
constexpr int EPI_WARPS = 8;
constexpr int TMEM_COLS = 2 * BN;
// pair mode: each CTA's stage holds its 128 rows of A and one 128-column
// half of B
constexpr int PAIR_B_BYTES = (BN / 2) * BK * 2;        // 16 KB
constexpr int PAIR_STAGE_BYTES = A_BYTES + PAIR_B_BYTES;  // 32 KB
constexpr int PAIR_STAGES = 6;
// row pairs per column sweep in FC1's grouped unit order
constexpr int kRowGroup = 8;

// Weight-gradient kernels stage their output in shared memory and write it
// with TMA stores.  Two configurations:
//  * skinny experts (few rows, one reduction block per 64 KB output tile):
//    the epilogue is the bottleneck, so one pipeline stage is traded for
//    double-buffered staging, two 32-row x 64-column boxes per epilogue warp
//    (128-byte swizzle);
//  * large experts (long reductions, tensor-bound): four stages and one
//    32 x 32 box per warp (64-byte swizzle).
// Each also keeps one box of zeros for experts with no rows.
template <GemmKind KIND, bool SKINNY, bool PAIR = false>
struct Cfg {
  static constexpr bool W = (KIND == GemmKind::kWgrad);
  static constexpr int stages = PAIR ? ((W && SKINNY) ? 4 : PAIR_STAGES) : (W && SKINNY) ? 3 : STAGES;
  static constexpr int stage_bytes = PAIR ? PAIR_STAGE_BYTES : STAGE_BYTES;
  // FC2 and FC1-dgrad store their bf16 output through one staged 32 x 32
  // box per epilogue warp (their reductions are short enough that plain
  // stores left the epilogue longer than the next tile's MMAs)
  static constexpr bool STO = (KIND == GemmKind::kFc2 || KIND == GemmKind::kDgrad ||
                               KIND == GemmKind::kFc1Act || KIND == GemmKind::kDgradAct);
  static constexpr int box_cols = SKINNY ? 64 : 32;
  static constexpr int box_bytes = 32 * box_cols * 2;
  static constexpr int nbuf = SKINNY ? 2 : 1;
  static constexpr int stg_bytes =
      W ? (nbuf * EPI_WARPS + 1) * box_bytes : (STO ? EPI_WARPS * box_bytes : 0);
};
template <GemmKind KIND, bool SKINNY, bool PAIR = false>
constexpr size_t smem_bytes(int E) {
  using C = Cfg<KIND, SKINNY, PAIR>;
  return 1024 /*align slack*/ + static_cast<size_t>(C::stages) * C::stage_bytes + C::stg_bytes +
         (2 * C::stages + 5) * 8 /*barriers*/ + 16 + 2 * (E + 1) * 4 /*scheduler*/;
}

// ------------------------------------------------------------ scheduling
struct Tile {
  int e;
  bool mc;      // 2-CTA unit that shares (multicasts) its B block
  int row0;     // ragged-row kinds: first global row of the tile
  int rows;     // ragged-row kinds: valid rows in the tile
  int m0;       // kWgrad: first output row (within the expert)
  int n0;       // first output column
  int kblocks;  // BK-blocks of the reduction
  int krow0;    // kWgrad: first row of the reduction (global)
  int klast;    // kWgrad: valid rows in the last reduction block
};

// Work units of a CL-CTA cluster.  With CL = 2 and at least two 128-row
// blocks, a unit is two consecutive row blocks sharing one 256-column block
// of B (CTA r takes row block 2i + r; each CTA fetches half of B and
// multicasts it).  An expert with a single row block (skinny experts of a
// fine-grained layer) pairs along N instead: CTA r takes column block 2i + r
// and loads everything itself, so no CTA of the pair sits idle.
template <GemmKind KIND>
__device__ __forceinline__ int row_blocks(const GemmArgs& g, const int* s_off, int e) {
  return (KIND == GemmKind::kWgrad) ? (g.R + BM - 1) / BM
                                    : (s_off[e + 1] - s_off[e] + BM - 1) / BM;
}
template <GemmKind KIND, int CL, bool PAIR = false>
__device__ __forceinline__ int tiles_of_expert(const GemmArgs& g, const int* s_off, int e) {
  const int nt = (g.N + BN - 1) / BN;
  const int mt = row_blocks<KIND>(g, s_off, e);
  if (PAIR) return ((mt + 1) / 2) * nt;   // 256-row units, also for one row block
  if (CL == 2 && mt == 1) return (nt + 1) / 2;
  return ((mt + CL - 1) / CL) * nt;
}

template <GemmKind KIND, int CL, bool PAIR = false>
__device__ __forceinline__ Tile decode_tile(const GemmArgs& g, const int* s_off,
                                            const int* s_ts, int t, int rank) {
  // expert e with s_ts[e] <= t < s_ts[e+1]
  int lo = 0, hi = g.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_ts[mid + 1] <= t) lo = mid + 1;
    else hi = mid;
  }
  Tile tl;
  tl.e = lo;
  const int local = t - s_ts[lo];
  const int nt = (g.N + BN - 1) / BN;
  int mi;
  if (!PAIR && CL == 2 && row_blocks<KIND>(g, s_off, lo) == 1) {
    tl.mc = false;
    mi = 0;
    tl.n0 = (2 * local + rank) * BN;
  } else {
    int pm, ni;
    if (g.col_major == 2) {
      // groups of kRowGroup row pairs, each group swept column-major
      const int np = (row_blocks<KIND>(g, s_off, lo) + CL - 1) / CL;
      const int grp = local / (kRowGroup * nt);
      const int idx = local - grp * (kRowGroup * nt);
      const int gg = min(kRowGroup, np - grp * kRowGroup);
      ni = idx / gg;
      pm = grp * kRowGroup + (idx - ni * gg);
    } else if (g.col_major) {
      const int np = (row_blocks<KIND>(g, s_off, lo) + CL - 1) / CL;
      ni = local / np;
      pm = local - ni * np;
    } else {
      pm = local / nt;
      ni = local - pm * nt;
    }
    tl.n0 = ni * BN;
    mi = CL * pm + rank;
    tl.mc = !PAIR && (CL == 2);
  }
  if constexpr (KIND == GemmKind::kWgrad) {
    tl.m0 = mi * BM;
    tl.krow0 = s_off[lo];
    const int kr = s_off[lo + 1] - s_off[lo];
    tl.kblocks = (kr + BK - 1) / BK;
    tl.klast = kr - (tl.kblocks - 1) * BK;
    tl.row0 = 0;
    tl.rows = 0;
  } else {
    tl.row0 = s_off[lo] + mi * BM;
    tl.rows = max(0, min(BM, s_off[lo + 1] - tl.row0));
    tl.kblocks = g.K / BK;
    tl.m0 = 0;
    tl.krow0 = 0;
    tl.klast = BK;
  }
  return tl;
}

// ------------------------------------------------------------ epilogues
__device__ __forceinline__ void st_global_v4(uint16_t* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// 32 fp32 accumulator columns -> 32 bf16 at p (64 bytes)
__device__ __forceinline__ void store_row32(uint16_t* p, const uint32_t (&r)[32]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    st_global_v4(p + 8 * v, pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                 pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                 pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                 pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
  }
}

template <GemmKind KIND, int ACT>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& g, const Tile& tl, int row_in_tile,
                                               int c, const uint32_t (&r)[32], float& amx) {
  const int col = tl.n0 + c * 32;  // first accumulator column of the chunk
  if (col >= g.N) return;
  if constexpr (KIND == GemmKind::kWgrad) {
    const int orow = tl.m0 + row_in_tile;
    if (orow >= g.R) return;
    uint16_t* p = g.out + static_cast<long long>(tl.e) * g.out_estride + orow * g.ldo + col;
    if (g.accumulate) {
      uint32_t a[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = r[i];
      add_bf16_row32(p, a);
      store_row32(p, a);
    } else {
      store_row32(p, r);
    }
  } else {
    if (row_in_tile >= tl.rows) return;
    const long long grow = tl.row0 + row_in_tile;
    if constexpr (KIND == GemmKind::kFc1Act) {
      if (g.out2) store_row32(g.out2 + grow * g.ldo2 + col, r);
      if constexpr (ACT == MOE_ACT_SRELU) {
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float h0 = fmaxf(__uint_as_float(r[2 * i]), 0.f);
          const float h1 = fmaxf(__uint_as_float(r[2 * i + 1]), 0.f);
          o[i] = pack_bf16x2(h0 * h0, h1 * h1);
          amx = fmaxf(amx, fmaxf(bf16_lo(o[i]), bf16_hi(o[i])));
        }
        uint16_t* p = g.out + grow * g.ldo + col;
#pragma unroll
        for (int v = 0; v < 4; ++v) st_global_v4(p + 8 * v, o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
      } else {
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float a0 = gate_phi<ACT>(__uint_as_float(r[4 * i + 0])) * __uint_as_float(r[4 * i + 1]);
          const float a1 = gate_phi<ACT>(__uint_as_float(r[4 * i + 2])) * __uint_as_float(r[4 * i + 3]);
          o[i] = pack_bf16x2(a0, a1);
          amx = fmaxf(amx, fmaxf(fabsf(bf16_lo(o[i])), fabsf(bf16_hi(o[i]))));
        }
        uint16_t* p = g.out + grow * g.ldo + col / 2;
        st_global_v4(p, o[0], o[1], o[2], o[3]);
        st_global_v4(p + 8, o[4], o[5], o[6], o[7]);
      }
    } else {  // kFc2, kDgrad
      store_row32(g.out + grow * g.ldo + col, r);
    }
  }
}

// FC2-dgrad + dActivation epilogue of one 32-column chunk of dA for the
// thread's row (all 32 lanes of the warp call it together).
//  * plain: r = dA; dH = act'(H; dA), same interleaving as H.
//  * routed (g.probs; [Sonic] "역전파 계산 그래프 재작성하기": the dH kernel
//    also emits dS and A' = S*A): r = dA' before the row's router
//    probability p; dH = act'(H; p dA'), A' = p act(H) (act recomputed from
//    the stored H); returns the chunk's part of <dA', act(H)>.
//  * with g.amax ([CuTe] "핵심 아이디어": the amax of the transposed,
//    Hadamard-rotated output is fused instead of a separate pass): each dH
//    column of the warp's 32 rows is rotated in two 16-row blocks by a
//    16-lane butterfly (H16 / 4) and its largest magnitude folded into amx.
//    Rows past the tile's valid rows count as zero; tiles start on an
//    expert's first row plus a multiple of 128, so the blocks run from each
//    expert's first row.
// 16 packed bf16 pairs of each lane's row into the warp's 32 x 32 box
// (64-byte swizzle: 16-byte chunk j of row r at j ^ ((r / 2) % 4)) and one
// TMA store of the box at (x, y); the box is reused once its previous store
// has read it.  Whole warps call it.
__device__ __forceinline__ void put_box32(uint8_t* box, const uint32_t* v, const CUtensorMap* m,
                                          int x, int y) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) bulk_wait_read_0();
  __syncwarp();
  uint8_t* row = box + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) =
        make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(m, box, x, y);
    bulk_commit();
  }
}

// box != nullptr: the warp's 32 rows all lie in the expert, and dH (tdh,
// [M_cap, ldo]) and A' (ta, [M_cap, ldo3]) leave through the warp's box and
// TMA stores instead of per-thread stores
template <int ACT>
__device__ __forceinline__ float dgrad_act_chunk(const GemmArgs& g, const Tile& tl, int row_in_tile,
                                                 int col, float p, const uint32_t (&r)[32],
                                                 float& amx, uint8_t* box = nullptr,
                                                 const CUtensorMap* tdh = nullptr,
                                                 const CUtensorMap* ta = nullptr) {
  constexpr bool GATED = (ACT != MOE_ACT_SRELU);
  constexpr int NV = GATED ? 64 : 32;  // dH values of the chunk
  const bool valid = row_in_tile < tl.rows;
  const bool routed = g.probs != nullptr;
  const long long grow = tl.row0 + row_in_tile;
  const int y0 = tl.row0 + (row_in_tile & ~31);   // the warp's first row (staged stores)
  float dh[NV];
  float ds = 0.f;
  if (valid) {
    uint32_t ap[16];  // routed: A' of the chunk's 32 dA columns, packed bf16 pairs
    uint32_t ob[16];  // staged: the box being filled
    if constexpr (!GATED) {
      const uint16_t* hp = g.aux + grow * g.ld_aux + col;
      uint16_t* pd = g.out + grow * g.ldo + col;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float h0 = fmaxf(bf16_lo(hw[i]), 0.f), h1 = fmaxf(bf16_hi(hw[i]), 0.f);
          float d0 = __uint_as_float(r[8 * v + 2 * i]), d1 = __uint_as_float(r[8 * v + 2 * i + 1]);
          if (routed) {
            const float a0 = h0 * h0, a1 = h1 * h1;
            ds += d0 * a0 + d1 * a1;
            ap[4 * v + i] = pack_bf16x2(p * a0, p * a1);
            d0 *= p;
            d1 *= p;
          }
          o[i] = pack_bf16x2(2.f * h0 * d0, 2.f * h1 * d1);
          dh[8 * v + 2 * i] = bf16_lo(o[i]);
          dh[8 * v + 2 * i + 1] = bf16_hi(o[i]);
        }
        if (box) {
#pragma unroll
          for (int i = 0; i < 4; ++i) ob[4 * v + i] = o[i];
          if (v == 3) put_box32(box, ob, tdh, col, y0);
        } else {
          st_global_v4(pd + 8 * v, o[0], o[1], o[2], o[3]);
        }
      }
    } else {
      const uint16_t* hp = g.aux + grow * g.ld_aux + 2 * col;
      uint16_t* pd = g.out + grow * g.ldo + 2 * col;
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint4 hv = *reinterpret_cast<const uint4*>(hp + 8 * v);
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};  // (gate, up) pairs
        uint32_t o[4];
        float a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float gg = bf16_lo(hw[i]), uu = bf16_hi(hw[i]);
          float da = __uint_as_float(r[4 * v + i]);
          float ph, dph;
          gate_phi_dphi<ACT>(gg, ph, dph);
          if (routed) {
            a[i] = ph * uu;
            ds += da * a[i];
            da *= p;
          }
          o[i] = pack_bf16x2(da * uu * dph, da * ph);
          dh[8 * v + 2 * i] = bf16_lo(o[i]);
          dh[8 * v + 2 * i + 1] = bf16_hi(o[i]);
        }
        if (routed) {
          ap[2 * v] = pack_bf16x2(p * a[0], p * a[1]);
          ap[2 * v + 1] = pack_bf16x2(p * a[2], p * a[3]);
        }
        if (box) {
#pragma unroll
          for (int i = 0; i < 4; ++i) ob[4 * (v & 3) + i] = o[i];
          if ((v & 3) == 3) put_box32(box, ob, tdh, 2 * col + 32 * (v >> 2), y0);
        } else {
          st_global_v4(pd + 8 * v, o[0], o[1], o[2], o[3]);
        }
      }
    }
    if (routed) {
      if (box) {
        put_box32(box, ap, ta, col, y0);
      } else {
        uint16_t* pa = g.out3 + grow * g.ldo3 + col;
#pragma unroll
        for (int v = 0; v < 4; ++v) st_global_v4(pa + 8 * v, ap[4 * v], ap[4 * v + 1], ap[4 * v + 2], ap[4 * v + 3]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < NV; ++i) dh[i] = 0.f;
  }
  if (g.amax != nullptr) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float x = dh[i];
#pragma unroll
      for (int sft = 1; sft < 16; sft <<= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, x, sft);
        x = (lane & sft) ? (o - x) : (x + o);
      }
      amx = fmaxf(amx, 0.25f * fabsf(x));
    }
  }
  return ds;
}

// FC1 epilogue with MXFP8 output: one 32-value block of A per call (64
// accumulator columns when gated, 32 for squared ReLU).  A is rounded to
// bf16 first; the codes quantise those bf16 values.
template <int ACT>
__device__ __forceinline__ void fc1_mx_block(const GemmArgs& g, const Tile& tl, int row_in_tile,
                                             int lane, int q, int cb, const uint32_t (&r0)[32],
                                             const uint32_t (&r1)[32], float& amx,
                                             uint8_t* box = nullptr,
                                             const CUtensorMap* th = nullptr,
                                             const CUtensorMap* ta = nullptr) {
  constexpr bool GATED = (ACT != MOE_ACT_SRELU);
  const int acc_col = tl.n0 + cb * (GATED ? 64 : 32);
  if (acc_col >= g.N) return;                       // uniform across the CTA
  const bool valid = row_in_tile < tl.rows;
  const long long grow = tl.row0 + row_in_tile;
  float a[32];
  if constexpr (GATED) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      a[i] = gate_phi<ACT>(__uint_as_float(r0[2 * i])) * __uint_as_float(r0[2 * i + 1]);
      a[16 + i] = gate_phi<ACT>(__uint_as_float(r1[2 * i])) * __uint_as_float(r1[2 * i + 1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float h = fmaxf(__uint_as_float(r0[i]), 0.f);
      a[i] = h * h;
    }
  }
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    pk[i] = pack_bf16x2(a[2 * i], a[2 * i + 1]);
    a[2 * i] = bf16_lo(pk[i]);
    a[2 * i + 1] = bf16_hi(pk[i]);
  }
  const int acol = GATED ? acc_col / 2 : acc_col;  // first A column of the block
  const int b = acol / 32;
  uint32_t qw[8];
  const uint32_t sc = mx_quant32(a, qw);
  if (box != nullptr) {
    // the warp's 32 rows all lie in the expert (MXFP8 experts are whole
    // 32-row blocks): H and A through the warp's box and TMA stores; the
    // transposed copy through the same box, rows written with a skew (row
    // r's 16-byte chunk j at (j + r/2) % 4, no bank conflicts either way)
    // so that lane c reads column c and quantises it as one 32 x 1 block
    const int y0 = tl.row0 + q * 32;
#pragma unroll
    for (int i = 0; i < 32; ++i) amx = fmaxf(amx, fabsf(a[i]));
    if (g.out2) {
      uint32_t hv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) hv[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
      put_box32(box, hv, th, acc_col, y0);
      if constexpr (GATED) {
#pragma unroll
        for (int i = 0; i < 16; ++i) hv[i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
        put_box32(box, hv, th, acc_col + 32, y0);
      }
    }
    put_box32(box, pk, ta, acol, y0);
    uint4* pq = reinterpret_cast<uint4*>(g.mx_q + grow * g.n_a + acol);
    pq[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    pq[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    const long long chunk = static_cast<long long>(tl.row0 / 32) * (g.n_a / 128) + b / 4;
    g.mx_s[chunk * 512 + mx_chunk_off(row_in_tile, b & 3)] = static_cast<uint8_t>(sc);
    if (g.mx_qT != nullptr) {
      if (lane == 0) bulk_wait_read_0();   // A's store has read the box
      __syncwarp();
      uint8_t* myrow = box + lane * 64;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(myrow + (((j + (lane >> 1)) & 3) * 16)) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      __syncwarp();
      float col[32];
      const int cj = lane >> 3, ce = (lane & 7) * 2;
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) {
        const uint16_t bv =
            *reinterpret_cast<const uint16_t*>(box + rr * 64 + (((cj + (rr >> 1)) & 3) * 16) + ce);
        col[rr] = __uint_as_float(static_cast<uint32_t>(bv) << 16);
      }
      __syncwarp();
      uint32_t cq[8];
      const uint32_t csc = mx_quant32(col, cq);
      uint4* pt = reinterpret_cast<uint4*>(g.mx_qT + static_cast<long long>(acol + lane) * g.M_cap + y0);
      pt[0] = make_uint4(cq[0], cq[1], cq[2], cq[3]);
      pt[1] = make_uint4(cq[4], cq[5], cq[6], cq[7]);
      g.mx_sT[static_cast<long long>(acol + lane) * (g.M_cap / 32) + y0 / 32] = static_cast<uint8_t>(csc);
    }
    return;
  }
  if (valid) {
#pragma unroll
    for (int i = 0; i < 32; ++i) amx = fmaxf(amx, fabsf(a[i]));
    uint16_t* pa = g.out + grow * g.ldo + acol;
#pragma unroll
    for (int v = 0; v < 4; ++v) st_global_v4(pa + 8 * v, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    if (g.out2) {
      store_row32(g.out2 + grow * g.ldo2 + acc_col, r0);
      if constexpr (GATED) store_row32(g.out2 + grow * g.ldo2 + acc_col + 32, r1);
    }
    uint4* pq = reinterpret_cast<uint4*>(g.mx_q + grow * g.n_a + acol);
    pq[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    pq[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    const long long chunk = static_cast<long long>(tl.row0 / 32) * (g.n_a / 128) + b / 4;
    g.mx_s[chunk * 512 + mx_chunk_off(row_in_tile, b & 3)] = static_cast<uint8_t>(sc);
  }
  // transposed copy: this warp's 32 rows form one column block
  if (g.mx_qT != nullptr && q * 32 < tl.rows) {
    uint32_t my_sc = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      uint32_t code;
      const uint32_t scj = mx_quant_lanes(a[j], code);
      g.mx_qT[static_cast<long long>(acol + j) * g.M_cap + grow] = static_cast<uint8_t>(code);
      if (lane == j) my_sc = scj;
    }
    g.mx_sT[static_cast<long long>(acol + lane) * (g.M_cap / 32) + grow / 32] =
        static_cast<uint8_t>(my_sc);
  }
}

// ------------------------------------------------------------ the kernel
template <GemmKind KIND, int ACT, bool MX, int CL, bool SKINNY, bool GATHER, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmD, const GemmArgs g) {
  constexpr bool A_MN = (KIND == GemmKind::kWgrad);
  constexpr bool B_MN = (KIND == GemmKind::kFc1Act || KIND == GemmKind::kFc2 ||
                         KIND == GemmKind::kWgrad);
  constexpr bool B_3D = (KIND != GemmKind::kWgrad);
  static_assert(!PAIR || (CL == 2 && !GATHER), "pair mode: TMA operands in 2-CTA clusters");
  // pair mode: one M = 256 MMA over both CTAs' rows
  constexpr uint32_t IDESC = idesc_bf16(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  using C = Cfg<KIND, SKINNY, PAIR>;
  constexpr int NST = C::stages;
  constexpr int SBYTES = C::stage_bytes;
  constexpr int BOX = C::box_bytes;
  constexpr int BOXC = C::box_cols;
  uint8_t* staging = smem + NST * SBYTES;                 // C::nbuf boxes per epilogue warp
  uint8_t* zero_box = staging + C::nbuf * EPI_WARPS * BOX;  // 32 x BOXC bf16 zeros
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + C::stg_bytes);
  uint64_t* empty_bar = full_bar + NST;
  uint64_t* tfull_bar = empty_bar + NST;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_ts = s_off + (g.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (CL == 2) ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit0 = blockIdx.x / CL;        // this cluster's first work unit
  const int unit_step = gridDim.x / CL;     // clusters in the grid
  constexpr uint16_t kPair = 0x3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      // gathered operands: lane 0's byte-count arrival plus one cp.async
      // arrival per producer lane.  Pair mode: the first CTA's full barrier
      // takes both CTAs' bytes; one commit (multicast) frees a stage in both
      mbar_init(&full_bar[i], GATHER ? 33 : 1);
      mbar_init(&empty_bar[i], PAIR ? 1 : CL);  // one commit from each CTA's MMA
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      // pair mode: the first CTA's MMA waits for both CTAs' epilogue warps
      mbar_init(&tempty_bar[i], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (KIND == GemmKind::kWgrad || (C::STO && g.tma_out)) prefetch_tmap(&tmC);
    if (KIND == GemmKind::kFc1Act || KIND == GemmKind::kDgradAct)
      if (g.tma_out) prefetch_tmap(&tmD);
  }
  if (KIND == GemmKind::kWgrad && warp >= 2) {  // epilogue threads clear the zero box
    for (int i = threadIdx.x - 64; i < BOX / 16; i += 32 * EPI_WARPS)
      reinterpret_cast<uint4*>(zero_box)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(tmem_slot, TMEM_COLS);
    else tmem_alloc(tmem_slot, TMEM_COLS);
  }
  if (warp == 2) {
    // offsets -> smem, made safe: non-decreasing and within [0, M_cap]
    bool bad = false;
    for (int i = lane; i <= g.E; i += 32) {
      int v = g.offsets[i];
      if (v < 0 || v > g.M_cap || (MX && (v & 31))) bad = true;
      s_off[i] = min(max(v, 0), g.M_cap);
      if (MX) s_off[i] &= ~31;
    }
    __syncwarp();
    if (lane == 0) {
      int prev = 0;
      for (int i = 0; i <= g.E; ++i) {
        if (s_off[i] < prev) { bad = true; s_off[i] = prev; }
        prev = s_off[i];
      }
      if (s_off[0] != 0) bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) set_err(g.err, MOE_DEV_BAD_OFFSETS);
    __syncwarp();
    // exclusive prefix of per-expert tile counts (warp scan, 32 experts a step)
    int carry = 0;
    for (int base = 0; base < g.E; base += 32) {
      const int e = base + lane;
      const int rows_e = (e < g.E) ? s_off[e + 1] - s_off[e] : 0;
      const bool owned = rows_e >= g.row_min && (g.row_max == 0 || rows_e < g.row_max);
      const int t = (e < g.E && owned) ? tiles_of_expert<KIND, CL, PAIR>(g, s_off, e) : 0;
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
  if constexpr (CL == 2) cluster_sync();   // peers' barriers initialised before any multicast
  else __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = s_ts[g.E];

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // B: with a 2-CTA cluster each CTA fetches half of the shared B block
    // and multicasts it into both CTAs' stage
    auto load_b = [&](uint8_t* sb, uint64_t* fb, const Tile& tl, int kb) {
      if constexpr (B_MN) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (tl.mc && (i >> 1) != rank) continue;
          uint8_t* dst = sb + i * MN_BOX_BYTES;
          const int kc = B_3D ? kb * BK : tl.krow0 + kb * BK;
          if (CL == 2 && tl.mc) {
            if constexpr (B_3D) tma_load_3d_mc(dst, &tmB, fb, tl.n0 + 64 * i, kc, tl.e, kPair);
            else tma_load_2d_mc(dst, &tmB, fb, tl.n0 + 64 * i, kc, kPair);
          } else {
            if constexpr (B_3D) tma_load_3d(dst, &tmB, fb, tl.n0 + 64 * i, kc, tl.e);
            else tma_load_2d(dst, &tmB, fb, tl.n0 + 64 * i, kc);
          }
        }
      } else {
        // K-major B: two 128-row halves
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (tl.mc && h != rank) continue;
          uint8_t* dst = sb + h * (B_BYTES / 2);
          if (CL == 2 && tl.mc) tma_load_3d_mc(dst, &tmB, fb, kb * BK, tl.n0 + 128 * h, tl.e, kPair);
          else tma_load_3d(dst, &tmB, fb, kb * BK, tl.n0 + 128 * h, tl.e);
        }
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_parity[NST];
    bool issued[NST];
    for (int i = 0; i < NST; ++i) { issued[i] = false; issued_parity[i] = 0; }
    bool ok = true;
    // token-tensor row of expert-major row r (gather_T, past the tensor, for
    // a pad row or a row past the expert)
    auto token_row = [&](long long r, bool valid) {
      const int p = (valid && r < g.M_cap) ? g.gather_pair[r] : -1;
      return p >= 0 ? p / g.gather_k : g.gather_T;
    };
    if constexpr (GATHER) {
      // gathered operand (the permute fused into the load, [Sonic] "Gather
      // Fusion"): the whole warp copies the token rows with 16-byte cp.async
      // into the 128-byte-swizzled layout a TMA load would give (row r's
      // chunk j at r*128 + (j ^ r%8)*16); one warp instruction moves four
      // 128-byte rows.  Lane l copies chunk l%8 of row 4i + l/8 in its i-th
      // copy; the token row indices it needs are held by lane (l & ~7) | i%8
      // in slot i/8 (rr[m] = row 4(l%8 + 8m) + l/8).  Each lane's copies
      // arrive on the full barrier (count 1 + 32); lane 0 waits, sets the
      // byte count of the other operand and loads it with TMA.
      const int ch = lane & 7, sub = lane >> 3;
      auto copy_row = [&](uint8_t* box, int row, int tok, int col0) {
        // zeros for a row past the tensor and for columns past its width
        // (a weight gradient's column block may lie past d)
        const bool ok_row = tok < g.gather_T && col0 + ch * 8 < g.gather_ld;
        const uint16_t* src = g.gather_src + (ok_row ? static_cast<long long>(tok) * g.gather_ld + col0 + ch * 8 : 0);
        cp_async16(box + row * 128 + ((ch ^ (row & 7)) * 16), src, ok_row ? 16u : 0u);
      };
      for (int t = unit0; t < total_tiles && ok; t += unit_step) {
        const Tile tl = decode_tile<KIND, CL, PAIR>(g, s_off, s_ts, t, rank);
        int rr[4];
        if constexpr (!A_MN) {
          // K-major A: the tile's 128 rows, the same in every stage
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int i = 4 * (ch + 8 * m) + sub;
            rr[m] = token_row(static_cast<long long>(tl.row0) + i, i < tl.rows);
          }
        }
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if constexpr (A_MN) {
            // weight gradient: the block's 64 reduction rows (those past the
            // expert read zeros)
            const int kmax = (kb == tl.kblocks - 1) ? tl.klast : BK;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const int i = 4 * (ch + 8 * m) + sub;
              rr[m] = token_row(static_cast<long long>(tl.krow0) + kb * BK + i, i < kmax);
            }
          }
          if (lane == 0) ok = mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          uint8_t* sa = smem + stage * SBYTES;
          uint8_t* sb = sa + A_BYTES;
          uint64_t* fb = &full_bar[stage];
          if constexpr (!A_MN) {
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, B_BYTES);
              load_b(sb, fb, tl, kb);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)
              copy_row(sa, 4 * i + sub, __shfl_sync(0xffffffffu, rr[i >> 3], (lane & ~7) | (i & 7)),
                       kb * BK);
          } else if (g.gather_operand == 0) {
            // A = the token tensor transposed: two 64-column boxes of the
            // block's 64 reduction rows
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, B_BYTES);
              load_b(sb, fb, tl, kb);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int box = i >> 4;
              copy_row(sa + box * MN_BOX_BYTES, 4 * (i & 15) + sub,
                       __shfl_sync(0xffffffffu, rr[(i & 15) >> 3], (lane & ~7) | (i & 7)),
                       tl.m0 + 64 * box);
            }
          } else {
            // B = the token tensor: four 64-column boxes; each CTA copies
            // all of them itself (no multicast of gathered rows)
            if (lane == 0) {
              mbar_arrive_expect_tx(fb, A_BYTES);
              const int kr = tl.krow0 + kb * BK;
              tma_load_2d(sa, &tmA, fb, tl.m0, kr);
              tma_load_2d(sa + MN_BOX_BYTES, &tmA, fb, tl.m0 + 64, kr);
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              const int box = i >> 4;
              copy_row(sb + box * MN_BOX_BYTES, 4 * (i & 15) + sub,
                       __shfl_sync(0xffffffffu, rr[(i & 15) >> 3], (lane & ~7) | (i & 7)),
                       tl.n0 + 64 * box);
            }
          }
          cp_async_arrive(fb);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
    } else if (PAIR && lane == 0) {
      // pair mode: this CTA's 128 rows of A and its 128-column half of B;
      // the bytes of both CTAs count on the first CTA's full barrier
      const uint32_t full0 = mapa_shared(smem_u32(&full_bar[0]), 0);
      for (int t = unit0; t < total_tiles && ok; t += unit_step) {
        const Tile tl = decode_tile<KIND, CL, PAIR>(g, s_off, s_ts, t, rank);
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * SBYTES;
          uint8_t* sb = sa + A_BYTES;
          const uint32_t fb = full0 + stage * 8;
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * SBYTES);
          if constexpr (A_MN) {
            // weight gradient: this CTA's 128 output rows of the activation^T
            const int kr = tl.krow0 + kb * BK;
            tma_load_2d_pair(sa, &tmA, fb, tl.m0, kr);
            tma_load_2d_pair(sa + MN_BOX_BYTES, &tmA, fb, tl.m0 + 64, kr);
          } else {
            tma_load_2d_pair(sa, &tmA, fb, kb * BK, tl.row0);
          }
          const int nh = tl.n0 + (BN / 2) * rank;   // this CTA's half of the tile's columns
          if constexpr (B_MN) {
            const int kc = B_3D ? kb * BK : tl.krow0 + kb * BK;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if constexpr (B_3D) tma_load_3d_pair(sb + i * MN_BOX_BYTES, &tmB, fb, nh + 64 * i, kc, tl.e);
              else tma_load_2d_pair(sb + i * MN_BOX_BYTES, &tmB, fb, nh + 64 * i, kc);
            }
          } else {
            tma_load_3d_pair(sb, &tmB, fb, kb * BK, nh, tl.e);
          }
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
    } else if (lane == 0) {
      for (int t = unit0; t < total_tiles && ok; t += unit_step) {
        const Tile tl = decode_tile<KIND, CL, PAIR>(g, s_off, s_ts, t, rank);
        for (int kb = 0; kb < tl.kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) { ok = false; break; }
          uint8_t* sa = smem + stage * SBYTES;
          uint64_t* fb = &full_bar[stage];
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          if constexpr (A_MN) {
            const int kr = tl.krow0 + kb * BK;
            tma_load_2d(sa, &tmA, fb, tl.m0, kr);
            tma_load_2d(sa + MN_BOX_BYTES, &tmA, fb, tl.m0 + 64, kr);
          } else {
            tma_load_2d(sa, &tmA, fb, kb * BK, tl.row0);
          }
          load_b(sa + A_BYTES, fb, tl, kb);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
    }
    if (!ok && lane == 0) {
      // give up: wait (bounded) for our copies in flight before exiting (in
      // pair mode the first CTA's full barriers count both CTAs' copies; the
      // second CTA waits a fixed 1 ms, far longer than a copy takes)
      if (PAIR && rank != 0) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {}
      } else {
        for (int i = 0; i < NST; ++i)
          if (issued[i]) {
            const uint32_t a = smem_u32(&full_bar[i]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(a, issued_parity[i]) && globaltimer_ns() - t0 < kWaitLimitNs) {}
          }
      }
    }
    __syncwarp();
  } else if (warp == 1 && (!PAIR || rank == 0)) {
    // ---------------------------------------------------------- MMA issuer
    // (pair mode: the first CTA's warp issues for both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int t = unit0; t < total_tiles && ok; t += unit_step, ++local) {
      const Tile tl = decode_tile<KIND, CL, PAIR>(g, s_off, s_ts, t, rank);
      const int buf = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      if (lane == 0)
        ok = PAIR ? mbar_wait_cluster(&tempty_bar[buf], aph ^ 1, abort_flag)
                  : mbar_wait(&tempty_bar[buf], aph ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      // One reduction block.  TAIL: an expert's ragged last block of a
      // weight gradient.  Its own instantiation keeps the tail's clearing
      // and fences out of the whole blocks' path: with them in the same
      // loop body, even untaken, the weight gradients' MMAs ran 12% slower.
      auto kblock = [&](int kb, auto tail_c) -> bool {
        constexpr bool TAIL = decltype(tail_c)::value;
        if (lane == 0) ok = mbar_wait(&full_bar[stage], phase, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        tc_fence_after();
        // rows gathered with cp.async were written through the generic proxy
        if (GATHER && lane == 0) fence_proxy_async_smem();
        uint8_t* sa = smem + stage * SBYTES;
        uint8_t* sb = sa + A_BYTES;
        int kk_n = BK / UK;
        if constexpr (TAIL) {
          // Only ceil(klast/16) MMAs touch the expert's rows; the rows after
          // klast up to that 16-row boundary belong to the next expert and
          // are cleared in all six 64x64 boxes (2 of A, 4 of B; pair mode: 2
          // of B in each CTA, the second CTA's written through the cluster)
          // before the MMAs read them.  Lane l clears 16-byte chunk l % 8 of
          // rows klast + l / 8, +4, ... in every box (a whole 128-byte row,
          // so the swizzle does not matter), with no division on this
          // per-tile path, which bounds the rate of skinny experts' tiles.
          kk_n = (tl.klast + UK - 1) / UK;
          const int zr = kk_n * UK - tl.klast;
          constexpr int NBOX = PAIR ? 4 : 6;
          if (zr > 0) {
            const int ch = lane & 7;
            for (int row = tl.klast + (lane >> 3); row < kk_n * UK; row += 4) {
#pragma unroll
              for (int box = 0; box < NBOX; ++box) {
                uint8_t* p = (box < 2 ? sa + box * MN_BOX_BYTES : sb + (box - 2) * MN_BOX_BYTES) +
                             row * 128 + ch * 16;
                *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0);
                if constexpr (PAIR) st_cluster_zero16(mapa_shared(smem_u32(p), 1));
              }
            }
            if constexpr (PAIR) {
              fence_proxy_async_cluster();
              fence_acq_rel_cluster();
            } else {
              fence_proxy_async_smem();
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
          auto mma = [&](int kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a0 + kk * 2048, MN_BOX_BYTES, 1024)
                                     : sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + kk * 2048, MN_BOX_BYTES, 1024)
                                     : sdesc_sw128(b0 + kk * 32, 16, 1024);
            if constexpr (PAIR) umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
            else umma_bf16(d_tmem, ad, bd, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          };
          if constexpr (TAIL) {
            for (int kk = 0; kk < kk_n; ++kk) mma(kk);
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / UK; ++kk) mma(kk);
          }
          if constexpr (PAIR) umma_commit_pair_mc(&empty_bar[stage]);      // frees it in both CTAs
          else if constexpr (CL == 2) umma_commit_mc(&empty_bar[stage], kPair);
          else umma_commit(&empty_bar[stage]);
        }
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1; }
        return true;
      };
      const bool ragged = KIND == GemmKind::kWgrad && tl.kblocks > 0 && tl.klast < BK;
      const int whole = ragged ? tl.kblocks - 1 : tl.kblocks;
      for (int kb = 0; kb < whole; ++kb)
        if (!kblock(kb, BoolC<false>{})) break;
      if constexpr (KIND == GemmKind::kWgrad)
        if (ok && ragged) kblock(tl.kblocks - 1, BoolC<true>{});
      if (!ok) break;
      if (lane == 0) {
        if constexpr (PAIR) umma_commit_pair_mc(&tfull_bar[buf]);   // both CTAs' epilogues
        else umma_commit(&tfull_bar[buf]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      // give up: let every MMA already issued finish before TMEM is freed
      if constexpr (PAIR) umma_commit_pair(drain_bar);
      else umma_commit(drain_bar);
      const uint32_t a = smem_u32(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
    __syncwarp();
  } else if (warp == 1) {
    // pair mode, second CTA: its MMA warp has nothing to issue
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;            // TMEM lane quadrant of this warp
    // pair mode: the first CTA's MMA warp waits for this CTA's epilogue too
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&tempty_bar[0]), 0) : 0u;
    const int wg = (warp - 2) >> 2;    // warpgroup: columns [wg*128, wg*128+128) of the tile
    const int row_in_tile = q * 32 + lane;
    int local = 0;
    uint32_t stg_slot = 0;
    float amx = 0.f;                   // NVFP4 statistic of this thread's outputs
    for (int t = unit0; t < total_tiles; t += unit_step, ++local) {
      const Tile tl = decode_tile<KIND, CL, PAIR>(g, s_off, s_ts, t, rank);
      const int buf = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&tfull_bar[buf], aph, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
      if constexpr (KIND == GemmKind::kFc1Act && MX) {
        constexpr int STEP = (ACT == MOE_ACT_SRELU) ? 32 : 64;
        // the warp's 32 rows in the expert: staged stores and transpose
        uint8_t* mbox = (g.tma_out && q * 32 < tl.rows) ? staging + (warp - 2) * BOX : nullptr;
        for (int cb = wg * (BN / STEP / 2); cb < (wg + 1) * (BN / STEP / 2); ++cb) {
          uint32_t r0[32], r1[32];
          tmem_ld32(tb + cb * STEP, r0);
          if constexpr (STEP == 64) tmem_ld32(tb + cb * STEP + 32, r1);
          tmem_wait_ld();
          fc1_mx_block<ACT>(g, tl, row_in_tile, lane, q, cb, r0, r1, amx, mbox, &tmC, &tmD);
        }
      } else if (KIND == GemmKind::kWgrad && tl.kblocks == 0 && g.accumulate) {
        // expert with no rows, accumulating: its weight gradient is untouched
      } else if (KIND == GemmKind::kWgrad && tl.m0 + q * 32 + 32 <= g.R && tl.kblocks == 0) {
        // expert with no rows: its weight gradient is zero; store the zero box
        if (lane == 0) {
          for (int c = wg * (128 / BOXC); c < (wg + 1) * (128 / BOXC); ++c) {
            const int col = tl.n0 + c * BOXC;
            if (col >= g.N) break;
            tma_store_3d(&tmC, zero_box, col, tl.m0 + q * 32, tl.e);
          }
          bulk_commit();
        }
        __syncwarp();
      } else if (KIND == GemmKind::kWgrad && tl.m0 + q * 32 + 32 <= g.R) {
        // whole 32-row slab valid: stage each 32-row box in shared memory
        // (swizzled like the tensor map) and let TMA write it with full-line
        // stores
        for (int c = wg * (128 / BOXC); c < (wg + 1) * (128 / BOXC); ++c) {
          const int col = tl.n0 + c * BOXC;
          if (col >= g.N) break;
          uint32_t r0[32], r1[32];
          tmem_ld32(tb + c * BOXC, r0);
          if constexpr (BOXC == 64) tmem_ld32(tb + c * BOXC + 32, r1);
          tmem_wait_ld();
          if (g.accumulate) {
            const uint16_t* op = g.out + static_cast<long long>(tl.e) * g.out_estride +
                                 static_cast<long long>(tl.m0 + q * 32 + lane) * g.ldo + col;
            add_bf16_row32(op, r0);
            if constexpr (BOXC == 64) add_bf16_row32(op + 32, r1);
          }
          uint8_t* buf = staging + ((warp - 2) * C::nbuf + (stg_slot % C::nbuf)) * BOX;
          if (lane == 0) {                     // the box is free once its last store read it
            if constexpr (C::nbuf == 2) bulk_wait_read_1();
            else bulk_wait_read_0();
          }
          __syncwarp();
          uint8_t* row = buf + lane * (BOXC * 2);
          // 128-byte swizzle: 16-byte chunk j of row r at j ^ (r % 8);
          // 64-byte swizzle: at j ^ ((r / 2) % 4)
          const int sw = (BOXC == 64) ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) = make_uint4(
                pack_bf16x2(__uint_as_float(r0[8 * j + 0]), __uint_as_float(r0[8 * j + 1])),
                pack_bf16x2(__uint_as_float(r0[8 * j + 2]), __uint_as_float(r0[8 * j + 3])),
                pack_bf16x2(__uint_as_float(r0[8 * j + 4]), __uint_as_float(r0[8 * j + 5])),
                pack_bf16x2(__uint_as_float(r0[8 * j + 6]), __uint_as_float(r0[8 * j + 7])));
            if constexpr (BOXC == 64)
              *reinterpret_cast<uint4*>(row + (((j + 4) ^ sw) * 16)) = make_uint4(
                  pack_bf16x2(__uint_as_float(r1[8 * j + 0]), __uint_as_float(r1[8 * j + 1])),
                  pack_bf16x2(__uint_as_float(r1[8 * j + 2]), __uint_as_float(r1[8 * j + 3])),
                  pack_bf16x2(__uint_as_float(r1[8 * j + 4]), __uint_as_float(r1[8 * j + 5])),
                  pack_bf16x2(__uint_as_float(r1[8 * j + 6]), __uint_as_float(r1[8 * j + 7])));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmC, buf, col, tl.m0 + q * 32, tl.e);
            bulk_commit();
          }
          ++stg_slot;
        }
      } else if (KIND == GemmKind::kWgrad && tl.kblocks == 0) {
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0;
        for (int c = wg * 4; c < wg * 4 + 4; ++c) epilogue_chunk<KIND, ACT>(g, tl, row_in_tile, c, z, amx);
      } else if constexpr (KIND == GemmKind::kDgradAct) {
        // this thread's row, the warpgroup's 128 columns (whole warps call
        // dgrad_act_chunk: the amax butterflies span the warp's rows)
        const bool vrow = row_in_tile < tl.rows;
        const long long grow = tl.row0 + row_in_tile;
        float p = 0.f, dsum = 0.f;
        if (g.probs != nullptr && vrow) {
          const int pr = g.pair_of_row[grow];
          p = pr >= 0 ? g.probs[pr] : 0.f;
        }
        // the warp's 32 rows all in the expert: staged TMA stores of dH (and A')
        uint8_t* box = (g.tma_out && q * 32 + 32 <= tl.rows) ? staging + (warp - 2) * BOX : nullptr;
        for (int c = wg * 4; c < wg * 4 + 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_wait_ld();
          const int col = tl.n0 + c * 32;
          if (col < g.N) dsum += dgrad_act_chunk<ACT>(g, tl, row_in_tile, col, p, r, amx, box, &tmC, &tmD);
        }
        const int half = tl.n0 + wg * 128;
        if (g.probs != nullptr && vrow && half < g.N) g.ds_part[grow * g.ds_parts + half / 128] = dsum;
      } else if (KIND == GemmKind::kFc1Act && g.tma_out && q * 32 + 32 <= tl.rows) {
        // FC1, the warp's 32 rows all in the expert: H (when saved) and A go
        // through the warp's 32 x 32 box (64-byte swizzle) and TMA stores.
        // Gated: a chunk of 32 accumulator columns gives 16 columns of A,
        // so A's box takes two chunks.
        uint8_t* box = staging + (warp - 2) * BOX;
        uint8_t* srow = box + lane * 64;
        const int sw = (lane >> 1) & 3;
        const int grow0 = tl.row0 + q * 32;
        auto put = [&](const uint32_t* v, const CUtensorMap* m, int x) {
          if (lane == 0) bulk_wait_read_0();     // the box's previous store has read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(srow + ((j ^ sw) * 16)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(m, box, x, grow0);
            bulk_commit();
          }
        };
        uint32_t av[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = wg * 4 + cc;     // cc's parity is c's: static indices into av
          const int col = tl.n0 + c * 32;
          if (col >= g.N) break;
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_wait_ld();
          if (g.out2) {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              hv[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            put(hv, &tmC, col);
          }
          if constexpr (ACT == MOE_ACT_SRELU) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = fmaxf(__uint_as_float(r[2 * i]), 0.f);
              const float h1 = fmaxf(__uint_as_float(r[2 * i + 1]), 0.f);
              av[i] = pack_bf16x2(h0 * h0, h1 * h1);
              amx = fmaxf(amx, fmaxf(bf16_lo(av[i]), bf16_hi(av[i])));
            }
            put(av, &tmD, col);
          } else {
            const int h = (cc & 1) * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float a0 = gate_phi<ACT>(__uint_as_float(r[4 * i + 0])) * __uint_as_float(r[4 * i + 1]);
              const float a1 = gate_phi<ACT>(__uint_as_float(r[4 * i + 2])) * __uint_as_float(r[4 * i + 3]);
              av[h + i] = pack_bf16x2(a0, a1);
              amx = fmaxf(amx, fmaxf(fabsf(bf16_lo(av[h + i])), fabsf(bf16_hi(av[h + i]))));
            }
            if (cc & 1) put(av, &tmD, (col - 32) / 2);
          }
        }
      } else if (C::STO && KIND != GemmKind::kFc1Act && g.tma_out && q * 32 + 32 <= tl.rows) {
        // the warp's 32 rows all lie in the expert: stage each 32 x 32 chunk
        // (64-byte swizzle: 16-byte chunk j of row r at j ^ ((r / 2) % 4))
        // and write it with a TMA store
        uint8_t* box = staging + (warp - 2) * BOX;
        for (int c = wg * 4; c < wg * 4 + 4; ++c) {
          const int col = tl.n0 + c * 32;
          if (col >= g.N) break;
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_wait_ld();
          if (lane == 0) bulk_wait_read_0();       // the box's previous store has read it
          __syncwarp();
          uint8_t* row = box + lane * 64;
          const int sw = (lane >> 1) & 3;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) = make_uint4(
                pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, box, col, tl.row0 + q * 32);
            bulk_commit();
          }
        }
      } else {
        for (int c = wg * 4; c < wg * 4 + 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_wait_ld();
          epilogue_chunk<KIND, ACT>(g, tl, row_in_tile, c, r, amx);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && rank != 0) mbar_arrive_cluster(tempty0 + buf * 8);
        else mbar_arrive(&tempty_bar[buf]);
      }
    }
    if ((KIND == GemmKind::kWgrad || C::STO) && lane == 0) bulk_wait_all();  // staged stores done
    if ((KIND == GemmKind::kFc1Act || KIND == GemmKind::kDgradAct) && g.amax != nullptr) {
      // non-negative floats order like their bit patterns
      const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(amx));
      if (lane == 0 && m != 0u) atomicMax(reinterpret_cast<unsigned int*>(g.amax), m);
    }
    __syncwarp();
  }

  tc_fence_before();
  // no CTA leaves while its peer may still multicast into it or arrive on it
  if constexpr (CL == 2) cluster_sync();
  else __syncthreads();
  if (*abort_flag && threadIdx.x == 0) set_err(g.err, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Cluster size of the grouped GEMM launches: pairs of CTAs share B tiles
// through TMA multicast.
constexpr int kCluster = 2;
constexpr int kMaxDevices = 64;

template <GemmKind KIND, int ACT, bool MX = false, bool SKINNY = false, bool GATHER = false,
          bool PAIR = false>
cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                     const CUtensorMap& td, const GemmArgs& g, int num_sms, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<KIND, ACT, MX, kCluster, SKINNY, GATHER, PAIR>;
  static_assert(smem_bytes<KIND, SKINNY, PAIR>(MOE_MAX_EXPERTS) <= 227 * 1024,
                "dynamic shared memory above the 227 KB a CTA may have");
  const size_t smem = smem_bytes<KIND, SKINNY, PAIR>(MOE_MAX_EXPERTS);
  // grid size and shared-memory attribute, set up once per device (a
  // process may drive several devices, one at a time)
  static int grid_of[kMaxDevices] = {0};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int& grid = grid_of[dev];
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(num_sms);
    q.blockDim = dim3(NUM_THREADS);
    q.dynamicSmemBytes = smem;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = kCluster;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &q);
    if (e != cudaSuccess) return e;
    const int most = num_sms / kCluster;
    grid = kCluster * ((clusters > 0 && clusters < most) ? clusters : most);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, td, g);
}

// ragged-row kind in pair mode or not, per activation
template <GemmKind KIND, bool MX, bool PAIR>
cudaError_t launch_act(int act, const CUtensorMap& ta, const CUtensorMap& tb,
                       const CUtensorMap& tc, const CUtensorMap& td, const GemmArgs& g,
                       int num_sms, cudaStream_t s) {
  switch (act) {
    case MOE_ACT_SWIGLU: return launch_t<KIND, MOE_ACT_SWIGLU, MX, false, false, PAIR>(ta, tb, tc, td, g, num_sms, s);
    case MOE_ACT_GEGLU: return launch_t<KIND, MOE_ACT_GEGLU, MX, false, false, PAIR>(ta, tb, tc, td, g, num_sms, s);
    case MOE_ACT_SRELU: return launch_t<KIND, MOE_ACT_SRELU, MX, false, false, PAIR>(ta, tb, tc, td, g, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

std::atomic<int> g_pair_mode{kPairAuto};

}  // namespace

int pair_mode() { return g_pair_mode.load(); }

int set_pair_mode(int mode) {
  if (mode < kPairNever || mode > kPairAlways) return -1;
  return g_pair_mode.exchange(mode);
}

bool use_pair(GemmKind kind, const GemmArgs& g) {
  if (g.gather_pair != nullptr) return false;
  const int m = g_pair_mode.load();
  if (m == kPairNever) return false;
  if (m == kPairAlways) return true;
  // experts of 256 rows or more on average: a 256-row unit rarely idles a
  // CTA, and the halved stages let six of them cover the load latency
  return static_cast<long long>(g.M_cap) >= static_cast<long long>(kPairRows) * g.E;
}

bool wgrad_skinny(const GemmArgs& g) {
  return static_cast<long long>(g.M_cap) < static_cast<long long>(kSkinnyRows) * g.E;
}

namespace {
// one launch in the given configuration (pair: 2-SM MMAs; skinny: the
// weight gradient's skinny-expert configuration, whose output box tc has)
cudaError_t launch_cfg(GemmKind kind, int act, const CUtensorMap& ta, const CUtensorMap& tb,
                       const CUtensorMap& tc, const CUtensorMap& td, const GemmArgs& g_in,
                       int num_sms, cudaStream_t s, bool mx, bool pair, bool skinny) {
  // Unit order: when an expert has no more row-pair units than column
  // tiles, sweep column tiles outermost, so that a wave of clusters reuses
  // each B column tile across the expert's row pairs while the A block stays
  // in L2; otherwise row pairs outermost.  Measured on the balanced layer
  // (E=8 x 4096 rows, d=8192, n=2048), column order against row order:
  // FC1-dgrad -4.7%, FC2-wgrad -1.4%, FC1 -1.2%, FC2 +2.0%; FC1-wgrad (32
  // row pairs, 16 column tiles) +1.6%, so it keeps row order.
  GemmArgs g = g_in;
  {
    const long long rows = (kind == GemmKind::kWgrad)
                               ? g.R
                               : (static_cast<long long>(g.M_cap) + g.E - 1) / (g.E > 0 ? g.E : 1);
    const long long units_m = ((rows + BM - 1) / BM + kCluster - 1) / kCluster;
    const long long nt = (g.N + BN - 1) / BN;
    g.col_major = units_m <= nt ? 1 : 0;
    // FC1 reads x over K = d (64 MB per expert on the balanced layer), more
    // than an L2 half keeps between two column sweeps: sweeping kRowGroup
    // row pairs at a time re-reads less of it (ncu, two balanced experts:
    // DRAM reads 678 -> 580 MB per launch; groups of 4 read 704 MB), at the
    // same speed
    if (kind == GemmKind::kFc1Act && units_m > kRowGroup) g.col_major = 2;
  }
  if (g.gather_pair != nullptr) {
    // the gathering producer is its own instantiation, so that the other
    // kernels keep their code and registers
    if (mx) return cudaErrorInvalidValue;
    if (kind == GemmKind::kWgrad)
      return skinny ? launch_t<GemmKind::kWgrad, 0, false, true, true>(ta, tb, tc, td, g, num_sms, s)
                             : launch_t<GemmKind::kWgrad, 0, false, false, true>(ta, tb, tc, td, g, num_sms, s);
#define MOE_GATHER_SWITCH(KIND)                                                                  \
  switch (act) {                                                                                 \
    case MOE_ACT_SWIGLU: return launch_t<KIND, MOE_ACT_SWIGLU, false, false, true>(ta, tb, tc, td, g, num_sms, s); \
    case MOE_ACT_GEGLU: return launch_t<KIND, MOE_ACT_GEGLU, false, false, true>(ta, tb, tc, td, g, num_sms, s);   \
    case MOE_ACT_SRELU: return launch_t<KIND, MOE_ACT_SRELU, false, false, true>(ta, tb, tc, td, g, num_sms, s);   \
    default: return cudaErrorInvalidValue;                                                       \
  }
    if (kind == GemmKind::kFc1Act) MOE_GATHER_SWITCH(GemmKind::kFc1Act)
    if (kind == GemmKind::kDgradAct) MOE_GATHER_SWITCH(GemmKind::kDgradAct)
#undef MOE_GATHER_SWITCH
    return cudaErrorInvalidValue;
  }
  if (mx) {
    if (kind != GemmKind::kFc1Act) return cudaErrorInvalidValue;
    return pair ? launch_act<GemmKind::kFc1Act, true, true>(act, ta, tb, tc, td, g, num_sms, s)
                             : launch_act<GemmKind::kFc1Act, true, false>(act, ta, tb, tc, td, g, num_sms, s);
  }
  if (pair) {
    switch (kind) {
      case GemmKind::kFc1Act: return launch_act<GemmKind::kFc1Act, false, true>(act, ta, tb, tc, td, g, num_sms, s);
      case GemmKind::kDgradAct: return launch_act<GemmKind::kDgradAct, false, true>(act, ta, tb, tc, td, g, num_sms, s);
      case GemmKind::kFc2: return launch_t<GemmKind::kFc2, 0, false, false, false, true>(ta, tb, tc, td, g, num_sms, s);
      case GemmKind::kDgrad: return launch_t<GemmKind::kDgrad, 0, false, false, false, true>(ta, tb, tc, td, g, num_sms, s);
      default: break;   // kWgrad: below
    }
  }
#define MOE_ACT_SWITCH(KIND)                                                         \
  switch (act) {                                                                     \
    case MOE_ACT_SWIGLU: return launch_t<KIND, MOE_ACT_SWIGLU>(ta, tb, tc, td, g, num_sms, s); \
    case MOE_ACT_GEGLU: return launch_t<KIND, MOE_ACT_GEGLU>(ta, tb, tc, td, g, num_sms, s);   \
    case MOE_ACT_SRELU: return launch_t<KIND, MOE_ACT_SRELU>(ta, tb, tc, td, g, num_sms, s);   \
    default: return cudaErrorInvalidValue;                                           \
  }
  switch (kind) {
    case GemmKind::kFc1Act: MOE_ACT_SWITCH(GemmKind::kFc1Act)
    case GemmKind::kDgradAct: MOE_ACT_SWITCH(GemmKind::kDgradAct)
    case GemmKind::kFc2: return launch_t<GemmKind::kFc2, 0>(ta, tb, tc, td, g, num_sms, s);
    case GemmKind::kDgrad: return launch_t<GemmKind::kDgrad, 0>(ta, tb, tc, td, g, num_sms, s);
    case GemmKind::kWgrad:
      if (pair)
        return skinny
                   ? launch_t<GemmKind::kWgrad, 0, false, true, false, true>(ta, tb, tc, td, g, num_sms, s)
                   : launch_t<GemmKind::kWgrad, 0, false, false, false, true>(ta, tb, tc, td, g, num_sms, s);
      return skinny ? launch_t<GemmKind::kWgrad, 0, false, true>(ta, tb, tc, td, g, num_sms, s)
                             : launch_t<GemmKind::kWgrad, 0, false, false>(ta, tb, tc, td, g, num_sms, s);
  }
#undef MOE_ACT_SWITCH
  return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_grouped_gemm(GemmKind kind, int act, const CUtensorMap& ta,
                                const CUtensorMap& tb, const CUtensorMap& tc, const GemmArgs& g,
                                int num_sms, cudaStream_t s, bool mx, const CUtensorMap* td_in,
                                int* launched) {
  const CUtensorMap& td = td_in ? *td_in : tc;
  if (launched) *launched = 1;
  if (g.gather_pair == nullptr && g.row_min == 0 && g.row_max == 0 && g.E > 1 &&
      g_pair_mode.load() == kPairAuto && !use_pair(kind, g)) {
    // A skinny layer's experts of kPairRows rows or more (hot experts of a
    // fine-grained layer) run first with the pair configuration, the rest
    // after them with the single-CTA one.  The two launches write disjoint
    // experts; experts with no rows belong to the second.
    GemmArgs gh = g;
    gh.row_min = kPairRows;
    GemmArgs gl = g;
    gl.row_max = kPairRows;
    const bool wl = (kind == GemmKind::kWgrad);
    cudaError_t e = launch_cfg(kind, act, ta, tb, (wl && td_in) ? *td_in : tc, td, gh, num_sms, s,
                               mx, true, wl && !td_in && wgrad_skinny(g));
    if (e != cudaSuccess) return e;
    if (launched) *launched = 2;
    return launch_cfg(kind, act, ta, tb, tc, td, gl, num_sms, s, mx, false, wgrad_skinny(g));
  }
  return launch_cfg(kind, act, ta, tb, tc, td, g, num_sms, s, mx, use_pair(kind, g),
                    wgrad_skinny(g));
}

}  // namespace moe
