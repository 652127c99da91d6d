/*
 * lcattn -- fused masked scaled-dot-product attention for GB300 (sm_103a).
 *
 * C ABI of the library liblcattn.so.  The operator is the one every kernel on
 * the pages benchmarks ("Long-Context Attention Benchmark: From Kernel
 * Efficiency to Distributed Context Parallelism", xllm-io blog review, sections
 * "密集注意力内核" and "稀疏注意力内核"): softmax attention under a mask, forward
 * and backward, bf16 inputs, head dim 128 (the pages' setting, section
 * "实验设置"), 64 or 256; MHA and GQA; an e4m3 forward at head dim 128.
 *
 *   S = scale * Q K^T,  P = row softmax over the allowed keys,  O = P V,
 *   LSE_i = ln sum_{j allowed} exp(S_ij)   (-inf for a row that allows nothing)
 *
 * The mask reaches the kernels as one of two descriptors:
 *   - column bounds (the column-wise representation the pages credit to
 *     FlashMask, section "掩码支持"): for every key column j, the allowed query
 *     rows are the union of two half-open intervals [a0,b0) and [a1,b1).  All
 *     twelve static mask families of the pages (section "注意力掩码模式") fit it.
 *   - block map (the dynamic Uniform Block / Variable Block masks, same
 *     section): a keep byte per (query block, key block) and query head, with
 *     arbitrary block boundaries.
 *
 * Conventions for every call:
 *   - Pointers marked "device" point to GPU memory, owned by the caller.  The
 *     library allocates nothing and frees nothing.  Between calls it keeps
 *     cached kernel attributes and, for lcattn_bwd_noalloc only, one fixed
 *     device array of LCATTN_NOALLOC_SCRATCH_BYTES per GPU (part of the
 *     library's image, held until the process exits) with its device address
 *     cached per GPU; that array's contents carry over from call to call.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream); the
 *     library never synchronises except in lcattn_read_status.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a negative status and launches nothing.
 *   - Tensors are bf16 (except LSE / D / accumulators, fp32) with the last
 *     dimension (head dim: 64, 128 or 256 elements) contiguous; the (batch, sequence,
 *     head) strides are given in elements and must be multiples of 8 (16
 *     bytes), and base pointers must be 16-byte aligned.  With B > 1 every
 *     batch stride must be at least the head dim (a zero, broadcast batch
 *     stride is refused with LCATTN_ERR_UNSUPPORTED); with B = 1 it is unused.
 *   - Query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 */
#ifndef LCATTN_H_
#define LCATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lcattn_stream_t; /* same handle as cudaStream_t */

/* ---- status codes ------------------------------------------------------ */
#define LCATTN_OK 0
#define LCATTN_ERR_INVALID_ARG (-1)   /* null pointer, bad size, bad stride      */
#define LCATTN_ERR_UNSUPPORTED (-2)   /* head dim, Hq % Hkv != 0, alignment         */
#define LCATTN_ERR_WORKSPACE (-3)     /* buffer smaller than the size query says  */
#define LCATTN_ERR_CUDA (-4)          /* a CUDA call or launch failed             */
#define LCATTN_ERR_DEVICE_TIMEOUT (-5)/* a kernel gave up waiting (bounded wait)  */
#define LCATTN_ERR_DEVICE_MASK (-6)   /* block offsets not increasing from 0 to S */
#define LCATTN_ERR_SCRATCH_LIMIT (-7) /* problem too large for lcattn_bwd_noalloc  */

/* ---- problem shape ------------------------------------------------------ */
typedef struct lcattn_shape {
  int64_t B;    /* batch                                                    */
  int64_t Sq;   /* query length                                             */
  int64_t Sk;   /* key length                                               */
  int64_t Hq;   /* query heads                                              */
  int64_t Hkv;  /* key/value heads; Hq % Hkv == 0                          */
  int64_t D;    /* head dim: 128, 64 or 256 (256: no deterministic
                 * backward; block selection and fp8: 128 only)             */
  /* element strides of (batch, sequence, head); the head dim is contiguous.
   * dO and dQ use q_stride's layout rules with o_stride / q_stride:
   *   O and dO share o_stride, Q and dQ share q_stride,
   *   K and dK share k_stride, V and dV share v_stride.                    */
  int64_t q_stride[3];
  int64_t k_stride[3];
  int64_t v_stride[3];
  int64_t o_stride[3];
} lcattn_shape;

/* ---- mask descriptor ----------------------------------------------------- */
#define LCATTN_MASK_COLBOUNDS 1
#define LCATTN_MASK_BLOCKMAP 2

typedef struct lcattn_mask_desc {
  int32_t kind;
  /* kind 1 (device) int32 [B][Sk][4] = {a0, b0, a1, b1}: query row i may attend
   * key column j iff a0 <= i < b0 or a1 <= i < b1.  Any int32 values are
   * allowed; intervals are clipped to [0, Sq).                              */
  const int32_t* col_bounds;
  /* kind 2 (device) uint8 [B][Hq][nQb][nKb]: nonzero = keep the block.       */
  const uint8_t* block_map;
  /* kind 2 (device) int32 [nQb+1] / [nKb+1]: block boundaries, nondecreasing,
   * first 0, last Sq (resp. Sk); checked on the device by the mask compiler. */
  const int32_t* q_block_offs;
  const int32_t* k_block_offs;
  int32_t nQb;
  int32_t nKb;
  /* kind 1, optional (device) int32 [B][Sq][4] = {c0, d0, c1, d1}: query row i
   * may attend key j iff c0 <= j < d0 or c1 <= j < d1 -- the same mask as
   * col_bounds, transposed (every static family of the pages has at most two
   * key intervals per row).  Any int32 values; intervals are clipped to
   * [0, Sk).  When given, the forward builds the row masks of partial tiles
   * from it (a few instructions per row instead of 128 column tests); tile
   * classification and the backward always use col_bounds.  The library cannot
   * check that the two forms agree: that is the caller's promise.  NULL = not
   * given.  16-byte aligned.                                                  */
  const int32_t* row_bounds;
} lcattn_mask_desc;

/* Tile classes written by the mask compiler (one byte per 128x128 tile). */
#define LCATTN_TILE_EMPTY 0
#define LCATTN_TILE_FULL 1
#define LCATTN_TILE_PARTIAL 2

/* Tile geometry: 128 query rows x 128 key columns. */
#define LCATTN_BLOCK_M 128
#define LCATTN_BLOCK_N 128

/* ---- tile metadata -------------------------------------------------------
 * The mask compiler turns a descriptor into per-tile classes and compacted
 * tile lists (section "掩码支持": FlashMask's column-wise representation exists to
 * skip masked-out work; here the skip decision is made once per 128x128 tile).
 * Layout of the buffer (all offsets from lcattn_tile_meta_layout):
 *   status  int32[4]                     device status words (0 = OK)
 *   sched   uint64[2]                    forward work counter and finished-CTA
 *                                        count (zero between calls; see lcattn_fwd)
 *   class   uint8 [B][nH][nQt][nKt]      LCATTN_TILE_* per tile
 *   fwd_cnt int32 [B][nH][nQt]           non-empty key tiles per query tile
 *   fwd_lst int32 [B][nH][nQt][nKt]      (kt << 1) | partial, kt increasing
 *   fwd_ord int32 [B][nH][nQt]           query tiles by fwd_cnt descending
 *   bwd_cnt int32 [B][nH][nKt]           non-empty query tiles per key tile
 *   bwd_lst int32 [B][nH][nKt][nQt]      (qt << 1) | partial, qt increasing
 *   bwd_ord int32 [B][nH][nKt]           key tiles by bwd_cnt descending
 * where nH = 1 for column bounds (the mask is the same for every head) and
 * nH = Hq for block maps.                                                    */
typedef struct lcattn_tile_meta_layout {
  int64_t nQt, nKt, nH, B;
  int64_t off_status, off_sched, off_class, off_fwd_cnt, off_fwd_lst, off_fwd_ord;
  int64_t off_bwd_cnt, off_bwd_lst, off_bwd_ord;
  int64_t total_bytes;
} lcattn_tile_meta_layout;

/* Fills *out for this shape and descriptor.  Returns a status. */
int lcattn_tile_meta_layout_of(const lcattn_shape* shape, const lcattn_mask_desc* mask,
                               lcattn_tile_meta_layout* out);

/* Bytes of device memory lcattn_mask_compile needs for `tile_meta`. */
size_t lcattn_tile_meta_size(const lcattn_shape* shape, const lcattn_mask_desc* mask);

/* Mask compiler.  Classifies every (query tile, key tile) pair as EMPTY, FULL
 * or PARTIAL, builds the forward (per query tile) and backward (per key tile)
 * lists of non-empty tiles and the longest-first orders.  `tile_meta` (device,
 * `bytes` >= lcattn_tile_meta_size) is overwritten.  The result depends only
 * on the shape's sizes and the descriptor, so one compile serves any number of
 * forward and backward calls with the same mask.                           */
int lcattn_mask_compile(const lcattn_shape* shape, const lcattn_mask_desc* mask,
                        void* tile_meta, size_t bytes, lcattn_stream_t stream);

/* ---- dynamic block selection -------------------------------------------
 * Builds the block map of a dynamic block-sparse mask from the activations:
 * the selection step the paper's peer reviews name for dynamic block-sparse
 * attention, blocks chosen by a TopK or a TopP criterion over pooled Q K^T
 * (tomesphere page for "Long-Context Attention Benchmark", section "Peer
 * Reviews"), producing the Uniform / Variable Block masks of the xllm-io blog
 * (section "注意力掩码模式").  The pages do not write the criterion out; the
 * library computes, for every batch b, query head h (KV head g = h / (Hq/Hkv))
 * and query block i:
 *   q_bar = mean of the query rows of block i (head h), k_bar[j] = mean of the
 *   key rows of block j (head g); an empty block's mean is 0;
 *   s[j] = scale * <q_bar, k_bar[j]>, written to `scores` when it is not NULL;
 *   candidates: both blocks non-empty and, if `causal`, k_offs[j] < q_offs[i+1];
 *   ranking: candidates by s descending, equal s by smaller j first;
 *   TOPK keeps the first min(top_k, #candidates) of the ranking;
 *   TOPP keeps a block while the softmax probability (over the candidates) of
 *   the blocks ranked before it sums to less than top_p, i.e. the shortest
 *   prefix of the ranking whose mass reaches top_p.
 * Arithmetic: block means and scores in fp32 (bf16 inputs, fp32 sums); the
 * TopK decision is exact on those fp32 scores; TopP's probabilities and
 * running mass are fp32, so a block whose mass-before lies within about
 * 1e-6 * #candidates of top_p may fall either way.                          */
#define LCATTN_SELECT_TOPK 1
#define LCATTN_SELECT_TOPP 2

typedef struct lcattn_select_desc {
  int32_t rule;    /* LCATTN_SELECT_TOPK or LCATTN_SELECT_TOPP                 */
  int32_t top_k;   /* TOPK: key blocks kept per (batch, head, query block), >= 0 */
  float top_p;     /* TOPP: mass threshold, finite; <= 0 keeps nothing, > 1 keeps
                    * every candidate                                          */
  int32_t causal;  /* 0 or 1 (see the candidate rule above)                    */
  /* device int32 [nQb+1] / [nKb+1]: block boundaries, the same arrays the
   * block-map descriptor takes.  Read clamped to [0, S] (block i covers
   * [clamp(offs[i]), max(clamp(offs[i]), clamp(offs[i+1])))) so that no read
   * leaves the tensors; offsets that are not nondecreasing from 0 to S give an
   * unspecified map, and lcattn_mask_compile reports them for the map.      */
  const int32_t* q_block_offs;
  const int32_t* k_block_offs;
  int32_t nQb;     /* 1 .. Sq                                                  */
  int32_t nKb;     /* 1 .. min(Sk, LCATTN_SELECT_MAX_KB)                       */
} lcattn_select_desc;

#define LCATTN_SELECT_MAX_KB 16384

/* Workspace (device bytes) lcattn_block_select needs: the fp32 block means
 * q_bar [B][Hq][nQb][128] and k_bar [B][Hkv][128][nKb] (transposed), each
 * 256-byte aligned; 0 for invalid input.                                    */
size_t lcattn_block_select_workspace_size(const lcattn_shape* shape, const lcattn_select_desc* sel);

/* Block selection.  q [B][Sq][Hq][128] and k [B][Sk][Hkv][128] bf16 (device,
 * head dim 128 only; LCATTN_ERR_UNSUPPORTED otherwise;
 * strides from `shape`; v/o strides unused) -> block_map uint8 [B][Hq][nQb][nKb]
 * (device, 1 = keep, 0 = drop; every byte written), ready for a block-map
 * descriptor with the same offsets.  `scores` (device fp32 [B][Hq][nQb][nKb])
 * is optional (NULL = not written).  `scale` > 0 is the softmax scale of the
 * scores (use the attention's).  Two kernels run in order on `stream`: the
 * block means (stage 1), then scores, ranking and selection (stage 2).     */
int lcattn_block_select(const lcattn_shape* shape, const void* q, const void* k,
                        const lcattn_select_desc* sel, float scale, uint8_t* block_map,
                        float* scores, void* workspace, size_t workspace_bytes,
                        lcattn_stream_t stream);

/* One stage of lcattn_block_select, same arguments (1 = block means,
 * 2 = scores and selection); any other stage returns LCATTN_ERR_INVALID_ARG. */
int lcattn_block_select_stage(int stage, const lcattn_shape* shape, const void* q, const void* k,
                              const lcattn_select_desc* sel, float scale, uint8_t* block_map,
                              float* scores, void* workspace, size_t workspace_bytes,
                              lcattn_stream_t stream);

/* Forward: the attention operator every dense and sparse kernel on the pages
 * computes ("Long-Context Attention Benchmark", xllm-io blog review, sections
 * "密集注意力内核" and "稀疏注意力内核"), restricted to the tiles the mask
 * compiler left non-empty; LSE is the per-row log-sum-exp that the pages'
 * distributed section ("分布式注意力机制", Ring P2P) merges partial results by.
 * q [B][Sq][Hq][D], k/v [B][Sk][Hkv][D] bf16 (device) ->
 * o [B][Sq][Hq][D] bf16 and lse [B][Hq][Sq] fp32 (natural log; -inf for a
 * row with no allowed key, whose O row is 0).  `tile_meta` must come from
 * lcattn_mask_compile with the same shape sizes and descriptor, and `mask`
 * is needed again because partial tiles evaluate the mask per element.
 * The kernel is persistent: its CTAs take query tiles, longest list first,
 * from a work counter in the scheduler words of `tile_meta`, and the last CTA
 * to run out of work puts the counter back to zero.  So forward calls that
 * share one `tile_meta` must not overlap in time (issue them on one stream);
 * after a DEVICE_TIMEOUT status, lcattn_clear_status also resets the counter.
 * The forward only reads the rest of `tile_meta`.  Part of every O tile is
 * written by TMA tensor stores through O's strides (the rest by plain
 * stores), so `o` must not overlap q, k or v; rows of padding between
 * sequences (a batch stride above Sq x the sequence stride) are never written. */
int lcattn_fwd(const lcattn_shape* shape, const void* q, const void* k, const void* v,
               const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* o,
               float* lse, lcattn_stream_t stream);

/* Forward with a workspace, for short query sides (the same operator as
 * lcattn_fwd, blog sections "密集注意力内核" / "稀疏注意力内核"; the split over
 * the key side is the flash-decoding scheme, merged by LSE).  When the regular
 * forward's work items (query tiles x head pairs x batch) are fewer than the
 * GPU's SMs -- decode-style rows, or a short chunk of queries against a long
 * key sequence (Sq < Sk, bottom-right aligned) -- and the mask is column
 * bounds, this call splits every query tile's key-tile list into slices that
 * run on separate SMs and merges them by their LSE (flash-decoding).  The
 * query heads of a GQA group share each K/V tile: they are packed into one
 * 128-row tile (Gp heads x 128/Gp positions, Gp the largest power of two
 * dividing Hq/Hkv, at most 128).  Otherwise it is exactly lcattn_fwd.
 * Same arguments and results as lcattn_fwd plus a workspace of
 * lcattn_fwd_workspace_size bytes (device, 16-byte aligned): fp32 per-slice
 * O / l [splits][B][Sq][Hq][D] and LSE [splits][B][Hq][Sq].  The split
 * count, and so the size, depends on the shape, the mask kind and the
 * current device's SM count; 0 means the call will not split (workspace may
 * then be NULL).  Two kernels run on `stream`: the slices, then the merge.  */
size_t lcattn_fwd_workspace_size(const lcattn_shape* shape, const lcattn_mask_desc* mask);
int lcattn_fwd_ws(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                  const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* o,
                  float* lse, void* workspace, size_t workspace_bytes, lcattn_stream_t stream);

/* FP8 forward: the same operator with e4m3 inputs (blog sections "密集注意力内核" /
 * "稀疏注意力内核"; the pages run bf16 and fix no fp8 semantics, so these are
 * the library's).  q [B][Sq][Hq][128], k and v [B][Sk][Hkv][128] hold OCP FP8
 * E4M3 codes (device, one byte per element; strides in elements = bytes, all
 * multiples of 16; 16-byte aligned); the real inputs are code * q_scale,
 * code * k_scale, code * v_scale (per-tensor factors > 0).  Head dim 128 only
 * (LCATTN_ERR_UNSUPPORTED otherwise).  Computes, per query row, with exact
 * fp32 logits scale * q_scale * k_scale * <q8, k8> and a running reference
 * m that moves to the row max whenever the max exceeds it by more than 4 (log2
 * units), so P = exp(logit - m) <= 16: P is quantized to e4m3 as 16 P for the
 * P V product (fp32 accumulation in tensor memory), l = sum of the
 * unquantized P, and o (bf16, o_stride, [B][Sq][Hq][128]) =
 * v_scale * (P8 V8) / (16 l) and lse = m + ln l are written (fp32
 * [B][Hq][Sq]; -inf and O = 0 for rows that allow nothing).  `tile_meta` from lcattn_mask_compile on the same shape and mask.
 * The workspace (lcattn_fwd_fp8_workspace_size bytes, 16-byte aligned) receives
 * V^T [B][Hkv][128][Skp] (e4m3, Skp = Sk rounded up to 16), written by a first
 * kernel so that both operands of the P V product are K-major (as
 * lcattn_fp8_transpose_v), and then holds the split-KV partials when the
 * shape takes that path (as lcattn_fwd_fp8_vt); the forward follows on
 * `stream`.  The size covers every mask of the shape.                     */
size_t lcattn_fwd_fp8_workspace_size(const lcattn_shape* shape);
int lcattn_fwd_fp8(const lcattn_shape* shape, const void* q, const void* k, const void* v, float q_scale,
                   float k_scale, float v_scale, const void* tile_meta, const lcattn_mask_desc* mask,
                   float scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                   lcattn_stream_t stream);

/* The two halves of lcattn_fwd_fp8, for callers that keep V transposed (an
 * e4m3 K/V cache written once and read by many decode steps, where a V^T
 * pass per step would double the V traffic of an HBM-bound forward).
 * lcattn_fp8_transpose_v writes vt = V^T [B][Hkv][128][Skp] e4m3 (contiguous,
 * lcattn_fp8_vt_size bytes, 16-byte aligned; keys in [Sk, Skp) zero) from v
 * (shape's v_stride).  lcattn_fwd_fp8_vt is the forward of lcattn_fwd_fp8 with
 * V given as vt.  Query sides that the bf16 forward would split over the key
 * list (lcattn_fwd_ws: decode rows, short query chunks; column bounds only)
 * take the same split-KV path here, with the same packing of a GQA group's
 * heads, and need lcattn_fwd_fp8_vt_workspace_size bytes of workspace for
 * the slices' partials (0: no workspace, which may then be NULL).  Errors as
 * for lcattn_fwd_fp8.                                                     */
size_t lcattn_fp8_vt_size(const lcattn_shape* shape);
int lcattn_fp8_transpose_v(const lcattn_shape* shape, const void* v, void* vt, lcattn_stream_t stream);
size_t lcattn_fwd_fp8_vt_workspace_size(const lcattn_shape* shape, const lcattn_mask_desc* mask);
int lcattn_fwd_fp8_vt(const lcattn_shape* shape, const void* q, const void* k, const void* vt, float q_scale,
                      float k_scale, float v_scale, const void* tile_meta, const lcattn_mask_desc* mask,
                      float scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                      lcattn_stream_t stream);

/* The backward calls below compute the gradients of the same operator (blog
 * sections "密集注意力内核" / "稀疏注意力内核"; the pages' sparse-kernel findings,
 * sections "稀疏内核性能" and "核心发现总结", single the backward out as the main
 * bottleneck).  They take head dim 64, 128 or 256; at 256 each dK/dV unit is
 * two CTAs, one per half of the head dim (the dK and dV accumulators of a
 * whole 128-key tile, 2 x 256 fp32 columns, do not fit in tensor memory beside
 * S and dP), and the deterministic backward returns LCATTN_ERR_UNSUPPORTED
 * with a workspace size of 0.
 *
 * Workspace (device bytes) lcattn_bwd needs: D = rowsum(dO * O) fp32
 * [B][Hq][Sq], the fp32 dQ accumulator [B][Hq][Sq][D] (head-major) and, when the dK/dV
 * work units (key tiles x KV heads x batch, times 2 at head dim 256) are too
 * few to fill the GPU in several waves -- under 1216, and the GQA group splits
 * evenly -- fp32 dK/dV
 * partials [2 or 4][2][B][Sk][Hkv][D]: each unit is split over 2 or 4
 * shares of its group's query heads and the partials are summed into dK, dV. */
size_t lcattn_bwd_workspace_size(const lcattn_shape* shape);

/* Backward of L = sum(O * dO) (blog sections "密集注意力内核" / "稀疏注意力内核":
 * the textbook gradients dV = P^T dO, dS = P * (dO V^T - rowsum(dO * O)),
 * dQ = scale * dS K, dK = scale * dS^T Q).  Inputs as for lcattn_fwd plus o, d_o (bf16,
 * o_stride) and lse from the forward.  Outputs dq (bf16, q_stride), dk
 * (k_stride) and dv (v_stride); dk/dv hold the sum over each GQA group.  The
 * three steps run in order on `stream`: D pre-pass (also zeroes the dQ
 * accumulator), one pass per key tile for dK/dV that adds dQ partials into the
 * accumulator, and the dQ conversion to bf16.                              */
int lcattn_bwd(const lcattn_shape* shape, const void* q, const void* k, const void* v,
               const void* o, const void* d_o, const float* lse, const void* tile_meta,
               const lcattn_mask_desc* mask, float scale, void* dq, void* dk, void* dv,
               void* workspace, size_t workspace_bytes, lcattn_stream_t stream);

/* One stage of lcattn_bwd (same operator and sections), same arguments: stage 1 = D pre-pass (and zeroing
 * of the dQ accumulator), 2 = dK/dV with dQ partials, 3 = dQ conversion.
 * Running stages 1, 2, 3 in order on one stream is exactly lcattn_bwd; the
 * stages exist so that each kernel can be scheduled or timed on its own.
 * Any other stage value returns LCATTN_ERR_INVALID_ARG.                   */
int lcattn_bwd_stage(int stage, const lcattn_shape* shape, const void* q, const void* k,
                     const void* v, const void* o, const void* d_o, const float* lse,
                     const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* dq,
                     void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     lcattn_stream_t stream);

/* Deterministic backward: the same gradients as lcattn_bwd (same arguments
 * and results), computed with no atomic or reduce-add anywhere, so that two
 * calls on the same inputs give identical bits.  dK and dV come from the
 * dK/dV pass without its dQ product; dQ comes from a pass of its own, one CTA
 * per (query tile, query head), that recomputes S = scale * Q K^T and
 * dP = dO V^T over the query tile's key list and accumulates dQ = dS K in
 * tensor memory (7 GEMMs per tile pair against lcattn_bwd's 5: measured 2-12%
 * slower, e.g. dense 8K 1018 against 1153 TFLOP/s).  Its workspace holds D
 * and, for split dK/dV units, their fp32 partials -- no fp32 dQ accumulator
 * (lcattn_bwd_deterministic_workspace_size bytes, smaller than lcattn_bwd's).
 * Three kernels in order on `stream` (D pre-pass, dK/dV, dQ), plus the
 * partials' sum when units are split.  Head dim 64 or 128.                 */
size_t lcattn_bwd_deterministic_workspace_size(const lcattn_shape* shape);
int lcattn_bwd_deterministic(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                             const void* o, const void* d_o, const float* lse, const void* tile_meta,
                             const lcattn_mask_desc* mask, float scale, void* dq, void* dk, void* dv,
                             void* workspace, size_t workspace_bytes, lcattn_stream_t stream);

/* Backward that allocates nothing and takes no workspace.  The pages have no
 * counterpart: this is an interface for callers that cannot hand the library
 * device memory of their own -- for example a plugin inside a host runtime that
 * owns every device allocation and forbids cudaMalloc (or offers no allocator
 * to its plugins), or a latency-critical serving path where cudaMalloc, which
 * may synchronise the device, is not allowed after start-up.
 *
 * Same arguments and results as lcattn_bwd without `workspace`.  The D vector
 * and the fp32 dQ accumulator live instead in one fixed device array inside the
 * library, LCATTN_NOALLOC_SCRATCH_BYTES (32 MiB) large; every GPU that loads
 * the library holds it until the process exits.  This call never splits
 * dK/dV work units (it needs no partials).  A problem whose D vector and dQ
 * accumulator exceed the array returns LCATTN_ERR_SCRATCH_LIMIT and launches
 * nothing.  The need is 4 * B*Hq*Sq bytes for D plus 4 * D * B*Hq*Sq bytes for
 * the accumulator, each rounded up to 256 bytes: 32 MiB covers B * Hq * Sq up
 * to 65,027 query rows at head dim 128 (e.g. 8 heads at 8K tokens) and
 * 129,055 at head dim 64.
 *
 * The first call on a device looks the array's device address up (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call on a device shares the one array and finds the previous
 * call's contents in it; the first stage of each call rewrites all of it that
 * must start at zero (the dQ accumulator) and all of D.  Calls whose work
 * overlaps on the GPU (different streams, different host threads) race on the
 * array and corrupt each other's gradients: order them on one stream.      */
#define LCATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int lcattn_bwd_noalloc(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                       const void* o, const void* d_o, const float* lse, const void* tile_meta,
                       const lcattn_mask_desc* mask, float scale, void* dq, void* dk, void* dv,
                       lcattn_stream_t stream);

/* ---- context parallelism by Ring P2P: the per-device building blocks -----
 * The pages' distributed half (xllm-io blog review, section "分布式注意力机制",
 * Ring P2P: several rounds of point-to-point exchange, overlapped with the
 * computation; the qualitative results are in section "分布式性能") splits the
 * sequence over devices.  Device r holds query shard r and K/V shard r; in
 * round t it computes its query shard against the K/V shard it holds, hands
 * that shard on to the next device, and merges the round's partial result
 * into its running one by log-sum-exp.  The backward walks the same ring:
 * each round adds the query shard's dQ terms locally and the K/V shard's dK/dV
 * terms into accumulators that travel with the shard back to its owner.
 * The calls below are what one device runs in one round; moving the shards
 * between devices is the caller's (any point-to-point transport into local
 * buffers).
 *
 * Shard descriptor: the mask of query rows [q0, q0 + Sq_s) against keys
 * [k0, k0 + Sk_s) of a global Sq x Sk problem (per batch entry), as a
 * descriptor of the Sq_s x Sk_s problem that lcattn_mask_compile and the
 * attention calls take.
 *   Column bounds (global->kind 1): col_bounds_out (device int32
 *   [B][Sk_s][4], 16-byte aligned) = clamp(col_bounds[b][k0 + j] - q0, 0,
 *   Sq_s) componentwise; if row_bounds_out is not NULL (global->row_bounds must
 *   then be given), row_bounds_out [B][Sq_s][4] = clamp(row_bounds[b][q0 + i] -
 *   k0, 0, Sk_s).  q_offs_out / k_offs_out are unused.
 *   Block maps (kind 2): q_offs_out [nQb+1] = clamp(q_block_offs - q0, 0, Sq_s)
 *   and k_offs_out [nKb+1] likewise; the map itself is reused as it is (same
 *   [B][Hq][nQb][nKb] array), the blocks outside the shard becoming empty.  The
 *   shard's descriptor must still have nQb <= Sq_s and nKb <= Sk_s.
 * One small kernel per output array on `stream`; LCATTN_ERR_INVALID_ARG for
 * shards outside the global problem or missing buffers.                     */
int lcattn_mask_shard(const lcattn_mask_desc* global, int64_t B, int64_t Sq, int64_t Sk,
                      int64_t q0, int64_t Sq_s, int64_t k0, int64_t Sk_s,
                      int32_t* col_bounds_out, int32_t* row_bounds_out,
                      int32_t* q_offs_out, int32_t* k_offs_out, lcattn_stream_t stream);

/* Merge of one round's partial forward result into the running result of a
 * query shard.  shape: the shard problem (B, Sq = query rows, Hq, D; its
 * o_stride is the layout of o_part and o_out).  o_acc (device fp32
 * [B][Sq][Hq][D], contiguous) and lse_acc ([B][Hq][Sq]) are the running
 * result; o_part (bf16) and lse_part ([B][Hq][Sq]) are the round's, from
 * lcattn_fwd on the shard pair.  With first = 1 the running result is set to
 * the part; otherwise, per row, with m = max(lse_acc, lse_part):
 *   o_acc <- (exp(lse_acc - m) o_acc + exp(lse_part - m) o_part) / (sum of the two weights),
 *   lse_acc <- m + ln(sum of the two weights),
 * and a row no round has allowed so far stays O = 0, LSE = -inf.  If o_out is
 * not NULL the merged O is also written there as bf16 (pass it in the last
 * round), with element strides o_out_stride (batch, sequence, head; NULL =
 * the shape's o_stride).  One kernel on `stream`.                          */
int lcattn_lse_merge(const lcattn_shape* shape, float* o_acc, float* lse_acc, const void* o_part,
                     const float* lse_part, void* o_out, const int64_t* o_out_stride, int first,
                     lcattn_stream_t stream);

/* Shard backward: lcattn_bwd's gradients of one shard pair, added into fp32
 * accumulators instead of written as bf16.  o and lse must be the query
 * shard's final (merged) O and LSE, so that P and D = rowsum(dO * O) are the
 * global ones.  dq_acc (device fp32 [B][Sq][Hq][D], contiguous) receives the
 * dQ terms of this key shard; dk_acc / dv_acc (fp32 [B][Sk][Hkv][D],
 * contiguous) receive the K/V shard's dK / dV terms from this query shard.
 * Nothing is zeroed: the caller clears the accumulators once.  The workspace
 * holds D only (lcattn_bwd_accum_workspace_size bytes).  Two kernels on
 * `stream` (the D pre-pass, then dK/dV with the dQ terms); head dim 64 or 128. */
size_t lcattn_bwd_accum_workspace_size(const lcattn_shape* shape);
int lcattn_bwd_accum(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                     const void* o, const void* d_o, const float* lse, const void* tile_meta,
                     const lcattn_mask_desc* mask, float scale, float* dq_acc, float* dk_acc,
                     float* dv_acc, void* workspace, size_t workspace_bytes, lcattn_stream_t stream);

/* fp32 [B][S][H][D] (device, contiguous) -> bf16 with element strides
 * dst_stride = (batch, sequence, head), e.g. the accumulated gradients of the
 * ring backward into dQ, dK, dV.  D is 64, 128 or 256.                      */
int lcattn_f32_to_bf16(const float* src, void* dst, int64_t B, int64_t S, int64_t H, int64_t D,
                       const int64_t dst_stride[3], lcattn_stream_t stream);

/* Synchronises `stream`, then returns the first nonzero device status word of
 * `tile_meta` (LCATTN_ERR_DEVICE_*), or LCATTN_OK.  Clears nothing.          */
int lcattn_read_status(const void* tile_meta, lcattn_stream_t stream);

/* Diagnostic: launches one CTA whose bounded device wait, on a barrier that
 * nothing completes, expires after about two seconds.  The kernel then records
 * LCATTN_ERR_DEVICE_TIMEOUT in the status words of `tile_meta` (device, any
 * buffer from lcattn_mask_compile) and returns, as every kernel of the library
 * does when one of its waits expires; the context stays usable.  Lets a caller
 * (or a test) exercise that path without faulting or hanging the GPU.  The
 * status words are only written, not cleared: clear them afterwards with
 * lcattn_clear_status.                                                      */
int lcattn_selftest_wait_timeout(void* tile_meta, lcattn_stream_t stream);

/* Zeroes the device status words of `tile_meta` (asynchronously). */
int lcattn_clear_status(void* tile_meta, lcattn_stream_t stream);

/* Static string for a status code. */
const char* lcattn_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int lcattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LCATTN_H_ */
