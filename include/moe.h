/*
 * moe.h - C ABI of libmoe, the GB300 (sm_103a) dropless MoE expert-MLP path.
 *
 * The path: a device-side routing layout (per-expert counts and prefix
 * offsets that never leave device memory), an expert-major permute, a
 * grouped FC1 GEMM with the gated activation applied in its epilogue, a
 * grouped FC2 GEMM, the combine, and the backward of all of these with the
 * activation derivative fused into the FC2-dgrad epilogue.
 *
 * Pages cited (title, section):
 *   [CuTe]  "NVIDIA CuTe DSL 융합 커널은 MoE 학습의 CPU·메모리 병목을 지운다"
 *   [Sonic] "SonicMoE로 보는 GPU 커널 최적화"
 *   [TE]    "NVIDIA Transformer Engine JAX dropless MoE 105→1,025 TFLOPs"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor argument is a DEVICE pointer owned by the caller.  Unless
 *    an entry point says otherwise the library allocates nothing, keeps no
 *    pointer after the call returns, and never synchronises the device or
 *    the stream: work is only enqueued on `stream` (a cudaStream_t passed as
 *    void*; NULL = legacy default stream).  No call copies anything to the
 *    host, so a whole forward + backward can be captured in a CUDA graph.
 *  - Layouts are row-major and dense (innermost dimension contiguous).
 *    bf16 tensors are passed as moe_bf16 (raw 16-bit patterns).
 *  - Pointers must be 16-byte aligned; d and n must be positive multiples
 *    of 64.
 *  - Return value: MOE_OK, or a negative MOE_E_* code for an error found
 *    on the host before anything is enqueued (null pointer, misalignment,
 *    unsupported size, CUDA launch failure).  Nothing is enqueued when a
 *    negative code is returned, except for MOE_E_CUDA, which reports the
 *    first failing launch.
 *  - Errors found on the device are OR-ed into the caller's int32 `err`
 *    word (MOE_DEV_* bits, sticky: the library never clears it).  No kernel
 *    traps; every wait inside a kernel is bounded in time and sets
 *    MOE_DEV_TIMEOUT when its limit runs out.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

/* host-side return codes */
#define MOE_OK 0
#define MOE_E_NULL (-1)        /* a required pointer is NULL            */
#define MOE_E_ALIGN (-2)       /* a pointer is not 16-byte aligned      */
#define MOE_E_SIZE (-3)        /* unsupported or inconsistent size      */
#define MOE_E_ARG (-4)         /* bad enum / flag value                 */
#define MOE_E_CUDA (-5)        /* CUDA runtime / launch error           */
#define MOE_E_WORKSPACE (-6)   /* workspace too small                   */

/* device-side error bits (OR-ed into *err) */
#define MOE_DEV_BAD_EXPERT 1   /* an expert id outside [-1, E) was skipped     */
#define MOE_DEV_OVERFLOW 2     /* rows past M_cap were dropped                  */
#define MOE_DEV_TIMEOUT 4      /* a bounded wait inside a kernel ran out        */
#define MOE_DEV_BAD_OFFSETS 8  /* offsets not non-decreasing within [0, M_cap];
                                  they were clamped before use                  */

/* activations ([CuTe] "무엇을 해결하려는가": SwiGLU, GeGLU, sReLU) */
#define MOE_ACT_SWIGLU 0       /* A_j = silu(H_2j) * H_2j+1                    */
#define MOE_ACT_GEGLU 1        /* A_j = gelu_tanh(H_2j) * H_2j+1               */
#define MOE_ACT_SRELU 2        /* A_j = max(H_j, 0)^2  (not gated)             */

/* flags */
#define MOE_FLAG_SAVE_H 1      /* forward also stores H (needed by backward)   */
#define MOE_FLAG_MXFP8 2       /* FC1 also emits MXFP8 A; FC2 is block-scaled
                                  MXFP8 (arguments in moe_mx_fwd)              */
#define MOE_FLAG_ACCUMULATE_DW 4 /* backward: dW1, dW2 += this step's weight
                                  gradients (gradient accumulation over
                                  micro-batches); experts with no rows keep
                                  their dW untouched                          */
#define MOE_FLAG_MX_SEPARATE_DH_QUANT 8 /* MXFP8 backward: quantise dH in its
                                  own pass after FC2-dgrad instead of in
                                  FC2-dgrad's epilogue (the unfused control;
                                  identical results)                          */

/*
 * MXFP8 data ([CuTe] "무엇을 해결하려는가" / "핵심 아이디어": an MXFP8 output
 * and its transposed copy written by the GEMM; [TE] "Transformer Engine이
 * 제공하는 세 가지 구성 요소": group-aware MXFP8 quantisation and an MXFP8
 * grouped GEMM).  Block rule (OCP MX v1.0): 32 values share a scale
 * X = 2^e, e = clamp(floor(log2 amax) - 8, -127, 127), stored as the E8M0
 * byte e + 127; each value is stored as E4M3(v / X), round to nearest even,
 * saturated to +-448.
 *
 * "MMA-tiled" scale layout: 128 rows (of A, or columns of W2) x 4
 * consecutive 32-blocks of the reduction index form one 512-byte chunk; the
 * scale of row r (0..127 inside the chunk) and block b (0..3) is byte
 * (r % 32) * 16 + (r / 32) * 4 + b.
 *   A scales:  chunk (g, c) at byte (g * (n/128) + c) * 512, where g =
 *              row0 / 32 for the 128-row tile [row0, row0+128) that holds
 *              the row (tiles start at offsets[e] + 128 i), c = block / 4.
 *              Size (M_cap/32) * (n/128) * 512 bytes.
 *   W2 scales: expert e, block b of rows (b = k / 32), column c: chunk
 *              (b/4, c/128) at byte e*(n/32)*d + ((b/4)*(d/128) + c/128)*512.
 *              Size E * (n/32) * d bytes.
 */
typedef struct moe_mx_fwd {
  const uint8_t* w2_q;  /* [E, n, d] E4M3 codes of W2 (moe_mx_quantize_weights) */
  const uint8_t* w2_s;  /* W2 scales, MMA-tiled                                   */
  uint8_t* a_q;         /* [M_cap, n] E4M3 codes of A, row-wise 1x32 blocks        */
  uint8_t* a_s;         /* A row-wise scales, MMA-tiled                            */
  uint8_t* a_qT;        /* [n, M_cap] codes of A^T, 32x1 blocks inside one expert,
                           or NULL (then a_sT is ignored)                          */
  uint8_t* a_sT;        /* [n, M_cap/32] E8M0 scales of a_qT                       */
  uint8_t* y_q;         /* GroupGemm + Quantize: [M_cap, d] codes of the bf16 Y,
                           row-wise 1x32 blocks, written by FC2's epilogue; or NULL */
  uint8_t* y_s;         /* [M_cap, d/32] E8M0 scales of y_q                        */
} moe_mx_fwd;

/*
 * MXFP8 backward ([TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩": the
 * fused GroupGemm + dActivation + Quantize/Transpose kernel; [CuTe]
 * "무엇을 해결하려는가": the transposed low-precision copy).  Every backward
 * GEMM takes MXFP8 operands whose 32-blocks run along its own reduction
 * index:
 *   FC2-dgrad + dAct  dY row-wise (blocks along d)  x  W2, blocks along d
 *   FC2-wgrad         A^T (the forward's transposed copy)  x  dY^T
 *   FC1-dgrad         dH row-wise (blocks along n1) x  W1, blocks along n1
 *   FC1-wgrad         x^T  x  dH^T
 * (transposed copies: 32-row blocks inside one expert).  dY, x and dH are
 * quantised inside moe_grouped_mlp_bwd_mx, into the caller's workspace.
 * "Weight tiles": W viewed as [rows, K] with blocks along K; 128 rows x 4
 * blocks per 512-byte chunk (byte layout as above), chunk (row/128) *
 * (K/128) + k/128; rows*K/32 bytes.
 */
typedef struct moe_mx_bwd {
  const uint8_t* a_qT;  /* [n, M_cap] codes of A^T (moe_mx_fwd.a_qT)             */
  const uint8_t* a_sT;  /* [n, M_cap/32] their scales (moe_mx_fwd.a_sT)          */
  const uint8_t* w2_q;  /* [E, n, d] codes of W2 with blocks along d
                           (moe_mx_quantize_weights_rowwise, rows = E*n)          */
  const uint8_t* w2_s;  /* weight tiles, E*n*d/32 bytes                            */
  const uint8_t* w1_q;  /* [E, d, n1] codes of W1 with blocks along n1
                           (rows = E*d)                                           */
  const uint8_t* w1_s;  /* weight tiles, E*d*n1/32 bytes                           */
  void* workspace;      /* device scratch, 256-byte aligned, owned by the caller   */
  size_t ws_bytes;      /* >= moe_mx_bwd_workspace_size(M_cap, d, n, act)          */
  uint8_t* dx_q;        /* GroupGemm + Quantize: [M_cap, d] codes of the bf16 dX,
                           row-wise 1x32 blocks, written by FC1-dgrad; or NULL      */
  uint8_t* dx_s;        /* [M_cap, d/32] E8M0 scales of dx_q                       */
} moe_mx_bwd;

/* Limits. */
#define MOE_MAX_EXPERTS 1024

/*
 * moe_router_topk - the router's selection: the top-k experts of each token
 * and the softmax of their logits ([TE] intro: a learned router activates
 * the top-K experts of each token; "Transformer Engine이 제공하는 세 가지
 * 구성 요소": gate, top-K, then dispatch).  The weighting is the softmax over
 * the k selected logits (the pages do not fix it).
 *   logits   [T, E] float32 (device).
 *   topk_idx [T, k] int32, written in decreasing logit order; ties go to the
 *            lower expert index.  The choice is exact and deterministic.
 *   probs    [T, k] float32, softmax of the selected logits.
 * Limits: 1 <= k <= E <= MOE_MAX_EXPERTS.
 */
int moe_router_topk(const float* logits, int T, int E, int k,
                    int32_t* topk_idx, float* probs, void* stream);

/*
 * moe_route_offsets - routing layout of the expert-major permuted buffer.
 *
 * Defined by [TE] "MoE 학습이 밀집 모델보다 어려운 이유: 래그드 텐서" (experts'
 * rows stored back to back in one ragged buffer), "용량 기반 MoE와 드롭리스
 * MoE" (dropless: no drop, no pad), "최적화 1: grouped GEMM" (per-expert
 * blocks aligned to a token unit; counts stay on the device) and
 * ""드롭리스"의 실제 경계" (one slot per (token, expert) pair, each expert
 * region padded to the alignment unit; a DROP policy that reports the
 * pre-truncation total).
 *
 *   topk_idx    [T, k] int32   expert of pair p = t*k + j; -1 = no route
 *                              (skipped silently); other ids outside [0, E)
 *                              are skipped and set MOE_DEV_BAD_EXPERT.
 *   align       >= 1           each expert's row count is rounded up to a
 *                              multiple of align (1 = no padding at all).
 *   M_cap                      rows of the permuted buffer; T*k + E*(align-1)
 *                              always suffices.
 * Outputs (device):
 *   counts      [E]   int32    pairs routed to each expert (before any drop).
 *   offsets     [E+1] int32    offsets[0] = 0, offsets[e+1] = offsets[e] +
 *                              roundup(counts[e], align), clamped to M_cap.
 *                              Rows of expert e: [offsets[e], offsets[e+1]).
 *   row_of_pair [T*k] int32    offsets[e] + rank of p among the pairs of e in
 *                              increasing p; -1 if skipped or dropped.
 *   pair_of_row [M_cap] int32  inverse of row_of_pair; -1 for pad and unused
 *                              rows.
 *   true_total  [1]   int32    rows demanded before truncation (the DROP
 *                              policy's true total); if it exceeds M_cap the
 *                              rows at or past M_cap are dropped and
 *                              MOE_DEV_OVERFLOW is set.
 *   workspace   device scratch of moe_route_workspace_size(T, k, E) bytes
 *               (contents need not be initialised; not kept after the call).
 * Every output is bit-exact and deterministic (no order depends on timing).
 * Limits: 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= E, T >= 0, 1 <= align <= 4096.
 */
size_t moe_route_workspace_size(int T, int k, int E);
int moe_route_offsets(const int32_t* topk_idx, int T, int k, int E, int align,
                      int M_cap, int32_t* counts, int32_t* offsets,
                      int32_t* row_of_pair, int32_t* pair_of_row,
                      int32_t* true_total, void* workspace, size_t ws_bytes,
                      int32_t* err, void* stream);

/*
 * moe_route_logits - the router fused into the routing layout ([TE]
 * "Transformer Engine이 제공하는 세 가지 구성 요소": gate, top-K selection,
 * dispatch and the grouped FFN form one fused block).  The top-k selection
 * and softmax of moe_router_topk run inside the layout's first pass, which
 * also counts each chosen pair, so no separate router launch is needed.
 *   logits [T, E] float32; writes topk_idx [T, k] and probs [T, k] (bit for
 *   bit what moe_router_topk writes) and the outputs of moe_route_offsets
 *   (counts, offsets, row_of_pair, pair_of_row, true_total), with the same
 *   workspace (moe_route_workspace_size), alignment, overflow and error
 *   rules.  Four launches (fill, fused select + count, scan, rank).
 */
int moe_route_logits(const float* logits, int T, int E, int k, int align, int M_cap,
                     int32_t* topk_idx, float* probs, int32_t* counts, int32_t* offsets,
                     int32_t* row_of_pair, int32_t* pair_of_row, int32_t* true_total,
                     void* workspace, size_t ws_bytes, int32_t* err, void* stream);

/*
 * moe_route_offsets_noalloc - moe_route_offsets for callers that cannot
 * allocate device memory.  The paper has no counterpart: this entry point
 * exists only for code that runs where cudaMalloc is off limits - inside a
 * CUDA-graph capture that must not grow a memory pool, under an
 * allocator-free runtime, or in a plugin whose host framework owns every
 * allocation and offers no scratch.  Same arguments and results as
 * moe_route_offsets, minus the workspace: the scratch is a fixed 1 MiB array
 * inside the library's device image (every GPU that loads the library holds
 * it until the process exits).
 *   - Limit: moe_route_workspace_size(T, k, E) =
 *     (ceil(T*k / 4096) + 1) * E * 4 bytes must be <= 1 MiB (E = 1024:
 *     T*k <= 1,044,480 pairs; E = 256: T*k <= 4,190,208); larger sizes
 *     return MOE_E_WORKSPACE and enqueue nothing.
 *   - The array's device address is looked up (cudaGetSymbolAddress, with
 *     the device current) on the first call in each CUDA context and cached
 *     under that context's unique ID.  A new context - a non-primary one,
 *     or the primary context that follows cudaDeviceReset - gets its own
 *     lookup on its first call.  Make that first call before any stream
 *     capture.
 *   - No cudaMalloc, cudaFree or allocating library call is made.  Nothing
 *     in the scratch needs to start at zero (each call writes every word it
 *     reads), but all calls share it: calls whose kernels can overlap on the
 *     GPU (different streams without ordering between them) race.
 */
int moe_route_offsets_noalloc(const int32_t* topk_idx, int T, int k, int E,
                              int align, int M_cap, int32_t* counts,
                              int32_t* offsets, int32_t* row_of_pair,
                              int32_t* pair_of_row, int32_t* true_total,
                              int32_t* err, void* stream);

/*
 * moe_permute - expert-major gather ([TE] "최적화 2: NCCL EP": dispatch
 * permutes the token rows; here without communication).
 *
 *   src [T, d] bf16, dst [M_cap, d] bf16.
 *   dst[r] = src[pair_of_row[r] / k]                 (scale == NULL, exact copy)
 *   dst[r] = bf16_rn(scale[p] * src[p / k]), p = pair_of_row[r]
 *                                                    (scale [T*k] float32; the
 *                                                    backward of the combine)
 *   dst[r] = 0 where pair_of_row[r] == -1 (pad and unused rows) or is
 *   otherwise outside [0, T*k).
 */
int moe_permute(const moe_bf16* src, const float* scale,
                const int32_t* pair_of_row, int T, int k, int d, int M_cap,
                moe_bf16* dst, void* stream);

/*
 * moe_permute_tokens - the same expert-major copy as moe_permute, walked in
 * token order ([TE] "최적화 2: NCCL EP"): each token row is read once and
 * written to each of its k rows, which moe_permute does by reading the token
 * row once per pair.  It takes both maps that moe_route_offsets writes.
 *
 *   src [T, d] bf16, dst [M_cap, d] bf16, scale [T*k] float32 or NULL,
 *   row_of_pair [T*k], pair_of_row [M_cap].
 *   For each pair p = t*k + j with r = row_of_pair[p] in [0, M_cap) and
 *   pair_of_row[r] == p:  dst[r] = src[t] (scale == NULL) or
 *   bf16_rn(scale[p] * src[t]).  dst[r] = 0 for every row r whose
 *   pair_of_row[r] lies outside [0, T*k).
 *   With the inverse pair of maps of moe_route_offsets this writes exactly
 *   what moe_permute writes, bit for bit; a row that pair_of_row assigns to
 *   a pair whose row_of_pair entry points elsewhere is left unwritten.
 *   Errors as moe_permute; row_of_pair may be NULL only when T == 0.
 */
int moe_permute_tokens(const moe_bf16* src, const float* scale,
                       const int32_t* row_of_pair, const int32_t* pair_of_row,
                       int T, int k, int d, int M_cap, moe_bf16* dst,
                       void* stream);

/*
 * moe_unpermute - combine ([TE] "최적화 2: NCCL EP": results return to token
 * order and each token accumulates its experts' outputs) and, optionally,
 * the router-score gradient ([Sonic] "역전파 계산 그래프 재작성하기":
 * dS_{t,e} = <dO_t, Y_{e,t}>).
 *
 *   src [M_cap, d] bf16 (expert-major rows), row_of_pair [T*k]; rows outside
 *   [0, M_cap) are treated like -1.
 *   If dst != NULL:   dst[t] = bf16_rn( sum_{j=0..k-1} w_tj * src[row(t,j)] ),
 *                     w = probs[t*k+j] (float32) or 1 when probs == NULL;
 *                     accumulated in float32 in increasing j; pairs with
 *                     row -1 contribute nothing.
 *   If dprobs != NULL: dprobs[t*k+j] = <dO[t], src[row(t,j)]> (float32; 0 for
 *                     row -1); dO [T, d] bf16 is then required.
 */
int moe_unpermute(const moe_bf16* src, const float* probs,
                  const int32_t* row_of_pair, int T, int k, int d, int M_cap,
                  moe_bf16* dst, const moe_bf16* dO, float* dprobs,
                  void* stream);

/*
 * moe_grouped_mlp_fwd - grouped expert MLP forward over ragged groups.
 *
 * [TE] "최적화 1: grouped GEMM" (one call over all experts with their real
 * row counts, no padding to a capacity, no device-to-host copy);
 * [CuTe] "핵심 아이디어 / 구조 / 동작 방식" (gate/up weight columns
 * interleaved so the GLU is computed in the GEMM epilogue and the 2n-wide
 * FC1 output need not be written).
 *
 * For each expert e, rows R_e = [offsets[e], offsets[e+1]) of x_perm:
 *   H_e = X_e W1_e         (float32 accumulation)
 *   A_e = act(H_e)         (from the float32 H; stored as bf16)
 *   Y_e = A_e W2_e         (A read back as bf16; stored as bf16)
 *
 *   x_perm  [M_cap, d] bf16       offsets [E+1] int32 (device, non-decreasing,
 *                                 offsets[E] <= M_cap)
 *   W1      [E, d, n1] bf16       n1 = 2n for gated acts, column 2j = gate_j,
 *                                 column 2j+1 = up_j; n1 = n for SRELU
 *   W2      [E, n, d]  bf16
 *   h_saved [M_cap, n1] bf16      written only with MOE_FLAG_SAVE_H (else may
 *                                 be NULL)
 *   a       [M_cap, n]  bf16      written
 *   y_perm  [M_cap, d]  bf16      written
 * Rows outside every expert's range are not written.  An expert with no
 * rows costs (almost) nothing.
 *
 * With MOE_FLAG_MXFP8 (`mx` required): FC1's epilogue also writes the
 * MXFP8 codes/scales of the bf16-rounded A (row-wise, and the transposed
 * copy if mx->a_qT != NULL), and FC2 computes Y_e from mx->a_q / a_s and
 * mx->w2_q / w2_s with block-scaled MXFP8 MMAs (W2 is then not read).
 * Requires n and d multiples of 128, M_cap a multiple of 32 and offsets
 * that are multiples of 32 (route with align = 32; otherwise
 * MOE_DEV_BAD_OFFSETS is set).
 *
 * amax_a (device float, or NULL): NVFP4's per-tensor statistic of the
 * forward output ([CuTe] "핵심 아이디어 / 구조 / 동작 방식": computed in the
 * GEMM instead of a separate memory pass).  The epilogue raises *amax_a to
 * max |A| over the bf16 A it writes (atomic maximum; the caller sets the
 * start value, e.g. 0).
 */
int moe_grouped_mlp_fwd(const moe_bf16* x_perm, const int32_t* offsets,
                        int E, int M_cap, int d, int n, const moe_bf16* W1,
                        const moe_bf16* W2, int act, int flags,
                        moe_bf16* h_saved, moe_bf16* a, moe_bf16* y_perm,
                        const moe_mx_fwd* mx, float* amax_a, int32_t* err,
                        void* stream);

/*
 * moe_grouped_mlp_bwd - backward of moe_grouped_mlp_fwd.
 *
 * The FC2-dgrad GEMM carries the activation derivative in its epilogue
 * ([CuTe] kernel family "GroupGemm + dActivation"; [Sonic] "GEMM
 * Overlapping": the dH kernel's epilogue reloads H and writes dH).
 * For each expert e:
 *   dA_e  = dY_e W2_e^T                     (float32, never stored)
 *   dH_e  = act'(H_e; dA_e)                 gated: dg = dA u phi'(g),
 *                                           du = dA phi(g); SRELU:
 *                                           dh = 2 max(h,0) dA  -> bf16
 *   dW2_e = A_e^T dY_e                      -> bf16
 *   dX_e  = dH_e W1_e^T                     -> bf16
 *   dW1_e = X_e^T dH_e                      -> bf16
 * An expert with no rows gets dW1_e = dW2_e = 0.
 *
 * flags: 0 or MOE_FLAG_ACCUMULATE_DW, gradient accumulation over
 * micro-batches (the training configuration's gradient_accumulation_steps,
 * [TE] "직접 재현하기: MaxText 컨테이너와 설정").  Accumulating, each weight
 * gradient becomes bf16(dW_old + X_e^T dH_e) (the old bf16 value is added
 * to the fp32 accumulator and the sum rounded once) and an expert with no
 * rows leaves its dW1_e, dW2_e untouched; dh and dx_perm are written as
 * usual.
 *
 *   x_perm [M_cap, d], h_saved [M_cap, n1], a [M_cap, n], dy_perm [M_cap, d]
 *   dh [M_cap, n1] (written), dx_perm [M_cap, d] (written),
 *   dW1 [E, d, n1] (written), dW2 [E, n, d] (written); all bf16.
 *
 * amax_dh (device float, or NULL): NVFP4's backward statistic, the amax of
 * the transposed, Hadamard-rotated dH, taken in the dH epilogue.  Per
 * expert, dH's rows are cut into 16-row blocks from the expert's first row
 * (the last one zero-padded) and each column of a block is multiplied by
 * the orthonormal 16x16 Hadamard matrix (Sylvester order, entries +-1/4);
 * *amax_dh is raised to the largest magnitude (atomic maximum; the caller
 * sets the start value).
 */
int moe_grouped_mlp_bwd(const moe_bf16* x_perm, const moe_bf16* h_saved,
                        const moe_bf16* a, const moe_bf16* dy_perm,
                        const int32_t* offsets, int E, int M_cap, int d,
                        int n, const moe_bf16* W1, const moe_bf16* W2,
                        int act, int flags, moe_bf16* dh, moe_bf16* dx_perm,
                        moe_bf16* dW1, moe_bf16* dW2, float* amax_dh,
                        int32_t* err, void* stream);

/*
 * moe_grouped_mlp_bwd_routed - backward with the router-score gradient
 * taken inside the expert MLP ([Sonic] "역전파 계산 그래프 재작성하기":
 * dS_{t,e} = <dO_t, Y_{e,t}> = <dO_t W2_e^T, A_e>, so Y is not needed; the
 * dH kernel's epilogue also emits dS and A' = S*A).
 *   do_perm [M_cap, d]: the gathered output gradient WITHOUT the router
 *   probability (moe_permute with scale = NULL); pair_of_row [M_cap] and
 *   probs [T*k] give each row's probability p (0 for pad rows).
 *   FC2-dgrad computes dA' = dO W2^T; its epilogue writes dh = act'(H; p dA'),
 *   a_scaled [M_cap, n] = p * act(H) (bf16) and ds_part [M_cap, ceil(n/128)]
 *   (fp32 partial <dA', act(H)> of each 128-column half tile, caller-owned
 *   scratch); FC2-wgrad then contracts a_scaled with do_perm.  dx_perm, dW1,
 *   dW2 and amax_dh as in moe_grouped_mlp_bwd.  Four GEMMs (each one or two
 *   launches, moe_set_pair_mma); finish with
 *   moe_router_grad_rows.  flags: 0 or MOE_FLAG_ACCUMULATE_DW (as in
 *   moe_grouped_mlp_bwd).  Errors as moe_grouped_mlp_bwd.
 */
int moe_grouped_mlp_bwd_routed(const moe_bf16* x_perm, const moe_bf16* h_saved,
                               const moe_bf16* do_perm, const int32_t* pair_of_row,
                               const float* probs, const int32_t* offsets, int E,
                               int M_cap, int d, int n, const moe_bf16* W1,
                               const moe_bf16* W2, int act, int flags, moe_bf16* dh,
                               moe_bf16* a_scaled, float* ds_part, moe_bf16* dx_perm,
                               moe_bf16* dW1, moe_bf16* dW2, float* amax_dh,
                               int32_t* err, void* stream);

/*
 * moe_grouped_mlp_bwd_routed_gather - moe_grouped_mlp_bwd_routed reading
 * the token tensors directly ([Sonic] "Gather Fusion": the gathered rows
 * are fetched again in the backward instead of being stored): FC2-dgrad's
 * dO rows, FC2-wgrad's dO rows and FC1-wgrad's x rows come from x [T, d]
 * and dO [T, d] through pair_of_row (token pair_of_row[r] / k; pad rows
 * read zeros), so neither permuted copy exists.  The other arguments, the
 * outputs (dh, a_scaled, ds_part, dx_perm in expert-major order; dW1, dW2)
 * and flags are those of moe_grouped_mlp_bwd_routed, and equal its results
 * on moe_permute(x), moe_permute(dO) bit for bit.  x and dO non-NULL and
 * 16-byte aligned even when T = 0.  Four GEMMs (the non-gathered ones may
 *   take two launches, moe_set_pair_mma); finish with
 * moe_router_grad_rows and moe_unpermute (dx).
 */
int moe_grouped_mlp_bwd_routed_gather(const moe_bf16* x, const moe_bf16* dO, int T, int k,
                                      const moe_bf16* h_saved, const int32_t* pair_of_row,
                                      const float* probs, const int32_t* offsets, int E,
                                      int M_cap, int d, int n, const moe_bf16* W1,
                                      const moe_bf16* W2, int act, int flags, moe_bf16* dh,
                                      moe_bf16* a_scaled, float* ds_part, moe_bf16* dx_perm,
                                      moe_bf16* dW1, moe_bf16* dW2, float* amax_dh,
                                      int32_t* err, void* stream);

/*
 * moe_router_grad_rows - dprobs [T*k] (fp32) of the routed backward
 * ([Sonic] "역전파 계산 그래프 재작성하기": dS = <dO W2^T, A>, whose partial sums
 * the FC2-dgrad epilogue leaves per 128-column half tile):
 * dprobs[p] = sum over the n_parts partials of ds_part's row row_of_pair[p]
 * (fixed order, so reruns are bitwise identical); 0 for pairs without a
 * row.  n_parts = ceil(n/128).  One launch.
 */
int moe_router_grad_rows(const float* ds_part, int n_parts, const int32_t* row_of_pair,
                         int T, int k, int M_cap, float* dprobs, void* stream);

/*
 * moe_mx_quantize_weights - MXFP8 copy of W2 for the block-scaled FC2
 * (blocks of 32 consecutive rows, FC2's reduction index, per column).
 *   W2 [E, n, d] bf16 -> w2_q [E, n, d] E4M3 codes, w2_s MMA-tiled scales
 *   (E * (n/32) * d bytes).  n, d multiples of 128.
 *   offsets: NULL, or the routing's device offsets [E+1]; then an expert
 *   with no rows (offsets[e+1] == offsets[e]) is skipped and its codes and
 *   scales are left as they were.  No GEMM of the layer reads an empty
 *   expert's weights, so a step that quantises its weights after routing
 *   ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소": the per-step
 *   MXFP8 cast of the expert weights) streams only the used experts.
 */
int moe_mx_quantize_weights(const moe_bf16* W2, int E, int n, int d,
                            const int32_t* offsets, uint8_t* w2_q, uint8_t* w2_s,
                            void* stream);

/*
 * moe_mx_quantize_weights2 - both MXFP8 copies of W2 that MXFP8 training
 * uses ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소": the MXFP8 cast
 * of the expert weights), from one read of W2: w2_q / w2_s as
 * moe_mx_quantize_weights (blocks
 * along n, for the forward FC2) and, if w2_q_rows != NULL, w2_q_rows
 * [E, n, d] / w2_s_rows (blocks along d, weight tiles: the
 * moe_mx_quantize_weights_rowwise layout with rows = E*n) for the
 * backward's FC2-dgrad.  Same sizes, offsets and errors as
 * moe_mx_quantize_weights.
 */
int moe_mx_quantize_weights2(const moe_bf16* W2, int E, int n, int d,
                             const int32_t* offsets, uint8_t* w2_q, uint8_t* w2_s,
                             uint8_t* w2_q_rows, uint8_t* w2_s_rows, void* stream);

/*
 * moe_mx_quantize_weights_rowwise - MXFP8 copy of a weight for a data
 * gradient ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소": the MXFP8
 * cast of the expert weights; here with blocks along the data gradient's
 * reduction index): W viewed as [rows, cols] bf16 (W2 [E, n, d] as rows = E*n,
 * cols = d; W1 [E, d, n1] as rows = E*d, cols = n1), blocks of 32 along
 * cols.  Writes q [rows, cols] codes and s in weight tiles (rows*cols/32
 * bytes).  rows, cols multiples of 128.
 *   offsets: NULL (E ignored), or the routing's device offsets [E+1] with
 *   rows = E * (rows per expert), rows per expert a multiple of 128
 *   (else MOE_E_SIZE); experts with no rows are skipped and left as they
 *   were, as in moe_mx_quantize_weights.
 */
int moe_mx_quantize_weights_rowwise(const moe_bf16* W, int rows, int cols,
                                    const int32_t* offsets, int E, uint8_t* q, uint8_t* s,
                                    void* stream);

/*
 * moe_mx_bwd_workspace_size - bytes of moe_mx_bwd.workspace for a layer
 * (0 for invalid sizes).  About M_cap * (3.4 d + 2.3 n1 + n/8).
 */
/*
 * moe_grouped_mlp_fwd_gather - moe_grouped_mlp_fwd with the permute fused
 * into FC1's operand load ([Sonic] "Gather Fusion": the up-projection
 * reads the routed rows itself, so the permuted copy of x, K times larger
 * than x, is never written): row r of
 * expert-major order is token pair_of_row[r] / k of x; pad rows
 * (pair_of_row[r] < 0) read zeros.
 *   x [T, d] bf16 (16-byte aligned, non-NULL even when T = 0: nothing is
 *   then read from it); pair_of_row [M_cap] as written by
 *   moe_route_offsets; the rest as moe_grouped_mlp_fwd.  flags: 0 or
 *   MOE_FLAG_SAVE_H (no MXFP8).  H, A, y_perm equal moe_grouped_mlp_fwd's
 *   on moe_permute(x) bit for bit.  Two GEMMs (FC2 may take two launches,
 *   moe_set_pair_mma).
 */
int moe_grouped_mlp_fwd_gather(const moe_bf16* x, int T, int k, const int32_t* pair_of_row,
                               const int32_t* offsets, int E, int M_cap, int d, int n,
                               const moe_bf16* W1, const moe_bf16* W2, int act, int flags,
                               moe_bf16* h_saved, moe_bf16* a, moe_bf16* y_perm,
                               float* amax_a, int32_t* err, void* stream);

/*
 * The unfused pieces of the expert MLP: a plain grouped GEMM and the
 * activation and its derivative as separate memory passes.  [CuTe]
 * "무엇을 해결하려는가" names the cost they carry (the activation reads the
 * FC1 output back and writes its result as its own memory pass) and
 * "공개된 근거에서 확인되는 점" the comparison the fused path is measured
 * against (grouped GEMM + activation kernels, unfused); the fused entry
 * points above replace them.  Each is one launch; the library allocates
 * nothing.
 *
 * moe_grouped_gemm - out_e = a_e B_e for the rows of each expert ([TE]
 * "최적화 1: grouped GEMM": one launch over the experts' ragged groups, the
 * counts read on the device).
 *   a [M_cap, K] bf16, offsets [E+1] (device, non-decreasing, offsets[E] <=
 *   M_cap), out [M_cap, N] bf16 (rows outside every expert not written).
 *   b_layout MOE_B_KN: B [E, K, N]; MOE_B_NK: B stored as [E, N, K] and
 *   out_e = a_e B_e^T.  K, N multiples of 64; pointers 16-byte aligned.
 *   Errors as moe_grouped_mlp_fwd.
 */
#define MOE_B_KN 0
#define MOE_B_NK 1
int moe_grouped_gemm(const moe_bf16* a, const int32_t* offsets, int E, int M_cap, int K,
                     int N, const moe_bf16* B, int b_layout, moe_bf16* out, int32_t* err,
                     void* stream);

/*
 * moe_activation - A = act(H) from a stored bf16 H [M_cap, n1] (n1 = 2n
 * gated, column 2j = gate_j, 2j+1 = up_j; n1 = n for MOE_ACT_SRELU) into
 * A [M_cap, n], over the rows below offsets[E].  The arithmetic is the FC1
 * epilogue's, applied to the bf16 H.
 * moe_activation_bwd - dH = act'(H; dA) (gated: dg = dA u phi'(g), du =
 * dA phi(g); SRELU: dh = 2 max(h, 0) dA) from bf16 H and dA [M_cap, n]
 * into dh [M_cap, n1], over the rows below offsets[E].
 *   n a multiple of 64; pointers 16-byte aligned.  Host errors as
 *   moe_grouped_mlp_fwd.
 */
int moe_activation(const moe_bf16* h, const int32_t* offsets, int E, int M_cap, int n,
                   int act, moe_bf16* a, void* stream);
int moe_activation_bwd(const moe_bf16* h, const moe_bf16* da, const int32_t* offsets, int E,
                       int M_cap, int n, int act, moe_bf16* dh, void* stream);

size_t moe_mx_bwd_workspace_size(int M_cap, int d, int n, int act);

/*
 * moe_mx_bwd_workspace_layout - where moe_grouped_mlp_bwd_mx keeps its
 * quantised operands inside mx->workspace, for callers that reuse them
 * (e.g. dH's MXFP8 copies) or check them.  Writes 11 byte offsets, in this
 * order: dY codes [M_cap, d] and scales (row tiles), dY^T codes [d, M_cap]
 * and scales (K tiles), x^T codes [d, M_cap] and scales (K tiles), A^T
 * scales re-tiled (K tiles), dH codes [M_cap, n1] and scales (row tiles),
 * dH^T codes [n1, M_cap] and scales (K tiles).  Valid after the call on the
 * stream has completed.  Host-only; returns the workspace size, 0 (and
 * writes nothing) on invalid sizes or a NULL offs.
 */
size_t moe_mx_bwd_workspace_layout(int M_cap, int d, int n, int act, size_t* offs);

/*
 * moe_set_pair_mma - how the grouped GEMMs (bf16 and block-scaled MXFP8)
 * pair the two CTAs of a cluster, process-wide:
 *   0  never: each CTA computes its own 128 x 256 tiles (1-SM MMAs; the two
 *      CTAs share B tiles through TMA multicast);
 *   1  automatic (the default): 2-SM MMAs over 256 x 256 tiles (each CTA
 *      loads 128 rows of A and half of B; tcgen05.mma.cta_group::2) when the
 *      average rows per expert, M_cap / E, reach 256; the block-scaled
 *      MXFP8 GEMMs other than the weight gradients always.  Below that
 *      average (E > 1) a GEMM makes two launches: the experts of 256 rows
 *      or more (weight gradients: reduction rows), found on the device,
 *      with 2-SM tiles, then the others as in mode 0;
 *   2  always 2-SM.
 * Results are identical across modes; the choice is for speed (and for
 * measuring one against the other).  Returns the previous mode, or
 * MOE_E_ARG for an unknown one.  Host-only; affects launches made after it.
 */
int moe_set_pair_mma(int mode);

/*
 * moe_workspace_size - device scratch for one layer's calls: the larger of
 * moe_route_workspace_size(T, k, E) and, when flags has MOE_FLAG_MXFP8,
 * moe_mx_bwd_workspace_size(M_cap, d, n, act).  One buffer of this size
 * serves both, since the routing layout and the MXFP8 backward use it at
 * different points of the step on the same stream; the other entry points
 * need no scratch.  Host-only, no CUDA call; 0 when every part is invalid.
 */
size_t moe_workspace_size(int T, int k, int E, int M_cap, int d, int n, int act, int flags);

/*
 * moe_grouped_mlp_bwd_mx - MXFP8 backward of the grouped expert MLP (same
 * results as moe_grouped_mlp_bwd up to MXFP8's rounding of the operands;
 * [TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩": GroupGemm +
 * dActivation + Quantize/Transpose; [CuTe] "무엇을 해결하려는가": the
 * transposed low-precision copy that the weight gradients read).
 *   x_perm [M_cap, d], h_saved [M_cap, n1], dy_perm [M_cap, d] bf16;
 *   offsets [E+1] multiples of 32 (route with align = 32); d, n multiples
 *   of 128, M_cap a multiple of 32.  Outputs dh [M_cap, n1], dx_perm
 *   [M_cap, d] (rows outside every expert untouched), dW1 [E, d, n1],
 *   dW2 [E, n, d] bf16 (zero for experts with no rows).  Seven launches:
 *   three quantisers (dY both ways, x transposed, A's scales re-tiled),
 *   FC2-dgrad + dAct + Quantize/Transpose (the epilogue writes the bf16 dH
 *   and both MXFP8 copies of it that FC1-dgrad and FC1-wgrad read, as the
 *   standalone tiled quantiser would, bit for bit), FC2-wgrad, FC1-dgrad,
 *   FC1-wgrad.  With MOE_FLAG_MX_SEPARATE_DH_QUANT, eight: FC2-dgrad + dAct
 *   stores dH alone and a separate pass quantises it.  In automatic pair
 *   mode each weight gradient of a layer below 256 rows per expert takes
 *   two launches (moe_set_pair_mma).
 *   flags: MOE_FLAG_ACCUMULATE_DW (as in moe_grouped_mlp_bwd),
 *   MOE_FLAG_MX_SEPARATE_DH_QUANT, or both.
 *   The quantised operands live in mx->workspace at the offsets
 *   moe_mx_bwd_workspace_layout gives.
 *   Errors: as moe_grouped_mlp_bwd; MOE_E_WORKSPACE if mx->ws_bytes is too
 *   small; offsets that are not multiples of 32 raise MOE_DEV_BAD_OFFSETS.
 */
int moe_grouped_mlp_bwd_mx(const moe_bf16* x_perm, const moe_bf16* h_saved,
                           const moe_bf16* dy_perm, const int32_t* offsets, int E,
                           int M_cap, int d, int n, int act, int flags,
                           const moe_mx_bwd* mx, moe_bf16* dh, moe_bf16* dx_perm,
                           moe_bf16* dW1, moe_bf16* dW2, int32_t* err, void* stream);

/*
 * moe_mx_quantize - group-aware MXFP8 quantisation of a ragged activation
 * ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소").
 *   src [rows, cols] bf16, offsets [E+1] (multiples of 32; rows at or past
 *   offsets[E] are not touched).  Writes q [rows, cols] codes with row-wise
 *   1x32 blocks and s [rows, cols/32] scales; and, if qT != NULL, the
 *   transposed copy qT [cols, rows] with column-wise 32x1 blocks inside one
 *   expert and sT [cols, rows/32].  cols, rows multiples of 32.
 */
int moe_mx_quantize(const moe_bf16* src, int rows, int cols,
                    const int32_t* offsets, int E, uint8_t* q, uint8_t* s,
                    uint8_t* qT, uint8_t* sT, int32_t* err, void* stream);

/*
 * moe_mx_quantize_tiled - moe_mx_quantize (the same group-aware
 * quantisation, [TE] "Transformer Engine이 제공하는 세 가지 구성 요소") with
 * the scales written in the layouts the block-scaled grouped GEMM reads, as
 * moe_grouped_mlp_bwd_mx
 * quantises its operands: s in row tiles (128-row tiles from offsets[e] +
 * 128 i, 512-byte chunks of 128 rows x 4 blocks, chunk (t0/32)*(cols/128) +
 * c/128 for the tile starting at row t0) and sT in reduction tiles (the
 * same tiles along the transposed copy's columns: chunk (t0/32)*(cols/128)
 * + c/128 holds columns c of the 128-column group x the tile's four 32-row
 * blocks).  Both buffers are rows*cols/8 bytes.  q may be NULL when qT is
 * given (transposed copy only), and qT NULL for the row-wise copy only.
 * Codes are those of moe_mx_quantize.  cols must be a multiple of 128
 * (MOE_E_SIZE otherwise), rows of 32; one warp covers 32 rows x 128
 * columns.
 */
int moe_mx_quantize_tiled(const moe_bf16* src, int rows, int cols,
                          const int32_t* offsets, int E, uint8_t* q, uint8_t* s,
                          uint8_t* qT, uint8_t* sT, int32_t* err, void* stream);

/*
 * Measurement hook (per host thread; no counterpart on the pages).
 * moe_set_launch_events(events, n): events points to n caller-created
 * cudaEvent_t handles (passed as void*).  From then on every grouped-GEMM
 * kernel launch, and every other entry-point call as a whole, records
 * events[2i] on its stream just before and events[2i+1] just after it, for
 * i = 0, 1, ... while 2i+1 < n; later launches record nothing.  The order
 * is the launch order: moe_grouped_mlp_fwd = FC1, FC2; moe_grouped_mlp_bwd
 * = FC2-dgrad+dAct, FC2-wgrad, FC1-dgrad, FC1-wgrad.  Passing (NULL, 0)
 * turns the hook off.  moe_launch_events_used() returns the number of
 * events recorded since the last moe_set_launch_events call.
 */
int moe_set_launch_events(void* const* events, int n);
int moe_launch_events_used(void);

/*
 * moe_selftest_bounded_wait - diagnostic (no counterpart on the pages).
 * Runs the bounded wait every kernel of the library uses on an mbarrier
 * that nothing arrives at, with a limit of limit_us microseconds
 * (1..1,000,000).  Expected outcome: MOE_DEV_TIMEOUT OR-ed into *err and
 * *waited_us >= limit_us; the device stays usable.  A completed barrier is
 * also waited on first and must not time out (else bit 16 is set).
 */
int moe_selftest_bounded_wait(int limit_us, int32_t* err, int32_t* waited_us,
                              void* stream);

/* Library version string (static storage). */
const char* moe_version(void);

/* Number of kernel launches the last successful call on this host thread
 * enqueued (for launch accounting; 0 before any call).  It includes the
 * second launch of each GEMM that automatic pair mode splits by expert
 * size (moe_set_pair_mma). */
int moe_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
