// Host layer of the C ABI declared in include/lcattn.h: argument validation,
// TMA descriptor encoding, tile-metadata layout, and the launches of the mask
// compiler, forward and backward kernels.  Allocates nothing.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "lcattn_internal.cuh"

using namespace lcattn;

namespace {

constexpr int64_t kMaxSeq = int64_t(1) << 20;  // tile lists and orders use int32 / smem sorts

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_shape(const lcattn_shape* s) {
  if (!s) return LCATTN_ERR_INVALID_ARG;
  if (s->B < 1 || s->Sq < 1 || s->Sk < 1 || s->Hq < 1 || s->Hkv < 1) return LCATTN_ERR_INVALID_ARG;
  if (s->Sq > kMaxSeq || s->Sk > kMaxSeq || s->B > 65535 || s->Hq > 65535)
    return LCATTN_ERR_UNSUPPORTED;
  if (s->D != 128 && s->D != 64 && s->D != 256) return LCATTN_ERR_UNSUPPORTED;
  if (s->Hq % s->Hkv != 0) return LCATTN_ERR_UNSUPPORTED;
  const int64_t* st[4] = {s->q_stride, s->k_stride, s->v_stride, s->o_stride};
  for (auto x : st)
    for (int i = 0; i < 3; ++i) {
      if (x[i] < 0) return LCATTN_ERR_INVALID_ARG;
      if (x[i] % 8 != 0) return LCATTN_ERR_UNSUPPORTED;  // 16-byte rows for TMA and vector I/O
    }
  // The head and sequence strides must at least separate rows.
  for (auto x : st)
    if (x[2] < s->D || x[1] < s->D) return LCATTN_ERR_INVALID_ARG;
  // With more than one batch entry, the batch stride must separate them too: a
  // zero stride (a broadcast view) would make the TMA and plain-load paths
  // disagree, and every output would have overlapping batch entries.  With
  // B = 1 the batch stride is never applied.
  if (s->B > 1)
    for (auto x : st)
      if (x[0] < s->D) return LCATTN_ERR_UNSUPPORTED;
  return LCATTN_OK;
}

int validate_mask(const lcattn_shape* s, const lcattn_mask_desc* m) {
  if (!m) return LCATTN_ERR_INVALID_ARG;
  if (m->kind == LCATTN_MASK_COLBOUNDS) {
    if (!m->col_bounds || !aligned16(m->col_bounds)) return LCATTN_ERR_INVALID_ARG;
    if (m->row_bounds && !aligned16(m->row_bounds)) return LCATTN_ERR_INVALID_ARG;
    return LCATTN_OK;
  }
  if (m->kind == LCATTN_MASK_BLOCKMAP) {
    if (!m->block_map || !m->q_block_offs || !m->k_block_offs) return LCATTN_ERR_INVALID_ARG;
    if (m->nQb < 1 || m->nKb < 1 || m->nQb > s->Sq || m->nKb > s->Sk) return LCATTN_ERR_INVALID_ARG;
    return LCATTN_OK;
  }
  return LCATTN_ERR_INVALID_ARG;
}

int layout_of(const lcattn_shape* s, const lcattn_mask_desc* m, lcattn_tile_meta_layout* L) {
  int st = validate_shape(s);
  if (st) return st;
  if ((st = validate_mask(s, m))) return st;
  std::memset(L, 0, sizeof(*L));
  L->B = s->B;
  L->nQt = (s->Sq + kBM - 1) / kBM;
  L->nKt = (s->Sk + kBN - 1) / kBN;
  L->nH = m->kind == LCATTN_MASK_BLOCKMAP ? s->Hq : 1;
  const int64_t bh = L->B * L->nH;
  int64_t off = 0;
  L->off_status = off;
  L->off_sched = off + 16; off = align_up(off + 32, 256);
  L->off_class = off;   off = align_up(off + bh * L->nQt * L->nKt, 256);
  L->off_fwd_cnt = off; off = align_up(off + 4 * bh * L->nQt, 256);
  L->off_fwd_lst = off; off = align_up(off + 4 * bh * L->nQt * L->nKt, 256);
  L->off_fwd_ord = off; off = align_up(off + 4 * bh * L->nQt, 256);
  L->off_bwd_cnt = off; off = align_up(off + 4 * bh * L->nKt, 256);
  L->off_bwd_lst = off; off = align_up(off + 4 * bh * L->nKt * L->nQt, 256);
  L->off_bwd_ord = off; off = align_up(off + 4 * bh * L->nKt, 256);
  L->total_bytes = off;
  return LCATTN_OK;
}

ProblemDev problem_of(const lcattn_shape* s) {
  ProblemDev p;
  p.B = (int)s->B; p.Sq = (int)s->Sq; p.Sk = (int)s->Sk;
  p.Hq = (int)s->Hq; p.Hkv = (int)s->Hkv; p.G = (int)(s->Hq / s->Hkv);
  p.D = (int)s->D;
  return p;
}

MaskDev mask_of(const lcattn_mask_desc* m) {
  MaskDev d;
  d.kind = m->kind;
  d.col_bounds = reinterpret_cast<const int4*>(m->col_bounds);
  d.row_bounds = m->kind == LCATTN_MASK_COLBOUNDS ? reinterpret_cast<const int4*>(m->row_bounds)
                                                  : nullptr;
  d.block_map = m->block_map;
  d.q_offs = m->q_block_offs;
  d.k_offs = m->k_block_offs;
  d.nQb = m->nQb;
  d.nKb = m->nKb;
  return d;
}

TileMetaDev meta_of(const lcattn_tile_meta_layout& L, const void* base) {
  uint8_t* p = static_cast<uint8_t*>(const_cast<void*>(base));
  TileMetaDev t;
  t.status = reinterpret_cast<int32_t*>(p + L.off_status);
  t.sched = reinterpret_cast<unsigned long long*>(p + L.off_sched);
  t.cls = p + L.off_class;
  t.fwd_cnt = reinterpret_cast<int32_t*>(p + L.off_fwd_cnt);
  t.fwd_lst = reinterpret_cast<int32_t*>(p + L.off_fwd_lst);
  t.fwd_ord = reinterpret_cast<int32_t*>(p + L.off_fwd_ord);
  t.bwd_cnt = reinterpret_cast<int32_t*>(p + L.off_bwd_cnt);
  t.bwd_lst = reinterpret_cast<int32_t*>(p + L.off_bwd_lst);
  t.bwd_ord = reinterpret_cast<int32_t*>(p + L.off_bwd_ord);
  t.nQt = (int)L.nQt; t.nKt = (int)L.nKt; t.nH = (int)L.nH; t.B = (int)L.B;
  return t;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [B][S][H][128] bf16 with element strides (b, s, h): 4-D map with a
// 64-element x box_h heads x box_s rows box (box_h * box_s = 128 rows of
// 128 bytes) and 128-byte swizzle (one K-major half tile per copy).
int encode_bshd_box(CUtensorMap* m, const void* ptr, int64_t B, int64_t S, int64_t H, int64_t D,
                    const int64_t st[3], uint32_t box_h, uint32_t box_s);

int encode_bshd(CUtensorMap* m, const void* ptr, int64_t B, int64_t S, int64_t H, int64_t D,
                const int64_t st[3]) {
  return encode_bshd_box(m, ptr, B, S, H, D, st, 1, 128);
}

int encode_bshd_box(CUtensorMap* m, const void* ptr, int64_t B, int64_t S, int64_t H, int64_t D,
                    const int64_t st[3], uint32_t box_h, uint32_t box_s) {
  auto fn = encode_fn();
  if (!fn) return LCATTN_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2,
                           (cuuint64_t)(st[0] > 0 ? st[0] : S * st[1]) * 2};
  cuuint32_t box[4] = {64, box_h, box_s, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LCATTN_OK : LCATTN_ERR_UNSUPPORTED;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LCATTN_OK : LCATTN_ERR_CUDA; }

// [B][S][H][128] e4m3 (one byte per element) with byte strides (b, s, h): a
// 4-D map with a 128-byte x 1 head x 128 rows box and 128-byte swizzle (one
// K-major 128 x 128 tile per copy).
int encode_bshd8(CUtensorMap* m, const void* ptr, int64_t B, int64_t S, int64_t H, const int64_t st[3],
                 uint32_t box_h = 1, uint32_t box_s = 128) {
  auto fn = encode_fn();
  if (!fn) return LCATTN_ERR_CUDA;
  cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2], (cuuint64_t)st[1], (cuuint64_t)(st[0] > 0 ? st[0] : S * st[1])};
  cuuint32_t box[4] = {128, box_h, box_s, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LCATTN_OK : LCATTN_ERR_UNSUPPORTED;
}

// V^T [B][Hkv][128][Skp] e4m3: box of 128 keys x 128 head-dim rows.
int encode_vt8(CUtensorMap* m, const void* ptr, int64_t B, int64_t Hkv, int64_t Skp) {
  auto fn = encode_fn();
  if (!fn) return LCATTN_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)Skp, 128, (cuuint64_t)Hkv, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)Skp, (cuuint64_t)(128 * Skp), (cuuint64_t)(Hkv * 128 * Skp)};
  cuuint32_t box[4] = {128, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LCATTN_OK : LCATTN_ERR_UNSUPPORTED;
}

int64_t fp8_skp(const lcattn_shape* s) { return align_up(s->Sk, 16); }

int64_t fwd8_ws_bytes(const lcattn_shape* s) { return align_up(s->B * s->Hkv * 128 * fp8_skp(s), 256); }

// The FP8 forward's extra rules: head dim 128, and every e4m3 row 16-byte
// aligned (strides in elements = bytes, multiples of 16).
int validate_fp8(const lcattn_shape* s) {
  if (s->D != 128) return LCATTN_ERR_UNSUPPORTED;
  const int64_t* st[3] = {s->q_stride, s->k_stride, s->v_stride};
  for (auto x : st)
    for (int i = 0; i < 3; ++i)
      if (x[i] % 16 != 0) return LCATTN_ERR_UNSUPPORTED;
  return LCATTN_OK;
}

// dK/dV work units (key tile, KV head, batch) are split over shares of the
// GQA group's query heads when there are too few units to fill the GPU in
// several waves (a partly empty last wave of equal units costs up to a wave);
// the shares' fp32 partials are summed afterwards.  Depends on the shape only,
// so the workspace size does too.
int bwd_parts(const lcattn_shape* s, int64_t nchunks = 1) {
  // (At head dim 256 every unit is two CTAs, one per half of the head dim.)
  const int64_t units = (s->Sk + kBN - 1) / kBN * s->Hkv * s->B * nchunks * (s->D == 256 ? 2 : 1);
  const int64_t G = s->Hq / s->Hkv;
  if (units < 304 && G % 4 == 0) return 4;
  if (units < 1216 && G % 2 == 0) return 2;
  return 1;
}

// Workspace: D [B][Hq][Sq], the fp32 dQ accumulator [B][Hq][Sq][D] and, for
// split units, the fp32 dK/dV partials [parts][2][B][Sk][Hkv][D]; with
// `chunk_room`, at least one such slot for the dK/dV accumulator of chunked
// units.
int64_t bwd_ws_bytes(const lcattn_shape* s, int parts, bool chunk_room) {
  const int64_t d_bytes = align_up(4 * s->B * s->Hq * s->Sq, 256);
  const int64_t acc_bytes = align_up(4 * s->B * s->Sq * s->Hq * s->D, 256);
  const int64_t slot = 2 * 4 * s->B * s->Sk * s->Hkv * s->D;
  const int64_t part_bytes = std::max<int64_t>(parts > 1 ? (int64_t)parts * slot : 0, chunk_room ? slot : 0);
  return d_bytes + acc_bytes + part_bytes;
}

// Workspace of the deterministic backward: D [B][Hq][Sq] and, for split units,
// the fp32 dK/dV partials [parts][2][B][Sk][Hkv][D] (no dQ accumulator).
int64_t bwd_det_ws_bytes(const lcattn_shape* s, int parts) {
  const int64_t d_bytes = align_up(4 * s->B * s->Hq * s->Sq, 256);
  const int64_t slot = 2 * 4 * s->B * s->Sk * s->Hkv * s->D;
  return d_bytes + (parts > 1 ? (int64_t)parts * slot : 0);
}

// Block maps carry one tile list per query head.  Units of one (key tile, KV
// head) walk every head's list in turn, and after a few waves the units in
// flight sit at unrelated heads and positions: their dQ reductions and Q/dO
// reads then spread over the whole group's rows and miss L2 (measured at 128K:
// 83% of the reduction sectors missed).  Such units are split into chunks of
// kChunkTiles query tiles, launched chunk-major, so that the units in flight
// share one chunk's rows.  Chunking pays from about 512 query tiles (64K
// tokens: +7%; 128K: +21%); at 256 the rows still fit and the extra per-unit
// work costs 8%.  Sizes measured: 16, 32, 64 and 128 tiles, 64 the fastest.
constexpr int64_t kChunkTiles = 64;
constexpr int64_t kChunkMinTiles = 512;
int64_t bwd_chunks(const lcattn_shape* s, const lcattn_mask_desc* m) {
  const int64_t nQt = (s->Sq + kBM - 1) / kBM;
  if (m->kind != LCATTN_MASK_BLOCKMAP || nQt < kChunkMinTiles) return 1;
  return (nQt + kChunkTiles - 1) / kChunkTiles;
}

}  // namespace

extern "C" {

int lcattn_tile_meta_layout_of(const lcattn_shape* shape, const lcattn_mask_desc* mask,
                               lcattn_tile_meta_layout* out) {
  if (!out) return LCATTN_ERR_INVALID_ARG;
  return layout_of(shape, mask, out);
}

size_t lcattn_tile_meta_size(const lcattn_shape* shape, const lcattn_mask_desc* mask) {
  lcattn_tile_meta_layout L;
  if (layout_of(shape, mask, &L) != LCATTN_OK) return 0;
  return (size_t)L.total_bytes;
}

int lcattn_mask_compile(const lcattn_shape* shape, const lcattn_mask_desc* mask, void* tile_meta,
                        size_t bytes, lcattn_stream_t stream) {
  lcattn_tile_meta_layout L;
  int st = layout_of(shape, mask, &L);
  if (st) return st;
  if (!tile_meta || !aligned16(tile_meta)) return LCATTN_ERR_INVALID_ARG;
  if (bytes < (size_t)L.total_bytes) return LCATTN_ERR_WORKSPACE;
  return cuda_status(launch_mask_compile(problem_of(shape), mask_of(mask), meta_of(L, tile_meta),
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int lcattn_fwd(const lcattn_shape* shape, const void* q, const void* k, const void* v,
               const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* o,
               float* lse, lcattn_stream_t stream) {
  lcattn_tile_meta_layout L;
  int st = layout_of(shape, mask, &L);
  if (st) return st;
  if (!q || !k || !v || !o || !lse || !tile_meta) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(tile_meta))
    return LCATTN_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !(scale < 1e30f)) return LCATTN_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, to;
  if ((st = encode_bshd(&tq, q, shape->B, shape->Sq, shape->Hq, shape->D, shape->q_stride))) return st;
  if ((st = encode_bshd(&tk, k, shape->B, shape->Sk, shape->Hkv, shape->D, shape->k_stride))) return st;
  if ((st = encode_bshd(&tv, v, shape->B, shape->Sk, shape->Hkv, shape->D, shape->v_stride))) return st;
  if ((st = encode_bshd(&to, o, shape->B, shape->Sq, shape->Hq, shape->D, shape->o_stride))) return st;
  FwdArgs a;
  a.pr = problem_of(shape);
  a.mask = mask_of(mask);
  a.meta = meta_of(L, tile_meta);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o = o;
  a.o_sb = shape->o_stride[0]; a.o_ss = shape->o_stride[1]; a.o_sh = shape->o_stride[2];
  a.lse = lse;
  return cuda_status(launch_fwd(tq, tk, tv, to, a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Plan for the packed / split-KV forward (short query sides, column bounds).
// It pays when packing the GQA group's heads into one tile needs at most half
// the (query tile, key tile) passes of the regular forward -- well under 128
// query rows per head -- or when the regular forward's items cannot fill the
// GPU and each walks a long key list.  The split count minimises a simple cost: waves of one CTA per SM
// times (a fixed cost of about four tiles for launch, pipeline fill and
// epilogue + the tiles of one slice).
struct SplitPlan {
  int splits = 0;  // 0: use the regular forward
  int Gp = 1, Rq = 128, nQc = 0;
};

SplitPlan split_plan(const lcattn_shape* s, const lcattn_mask_desc* m) {
  SplitPlan p;
  if (m->kind != LCATTN_MASK_COLBOUNDS) return p;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0)
    return p;
  const int64_t G = s->Hq / s->Hkv;
  const int64_t nQt = (s->Sq + kBM - 1) / kBM, nKt = (s->Sk + kBN - 1) / kBN;
  if (nKt < 4) return p;
  const int gp = split_heads_packed((int)G);
  const int64_t rq = 128 / gp;
  const int64_t nqc = (s->Sq + rq - 1) / rq;
  const int64_t passes_regular = s->Hq * nQt, passes_packed = s->Hq / gp * nqc;
  const int64_t hpc = G % 2 == 0 ? 2 : 1;
  const int64_t items = s->Hq / hpc * s->B * nQt;
  // Filling idle SMs pays only when each item has a long key list (at 8 key
  // tiles the slices' merge costs more than the idle SMs: 1K causal, 105 ->
  // 90 TFLOP/s forward when split).
  const bool packs = 2 * passes_packed <= passes_regular;
  const bool fills = items < nsm && nKt >= 16;
  if (!packs && !fills) return p;
  const int64_t base = s->B * s->Hkv * (G / gp) * nqc;
  const int64_t max_splits = std::max<int64_t>(1, std::min<int64_t>(64, nKt / 4));
  int64_t best = 1;
  double best_cost = 0.0;
  for (int64_t k = 1; k <= max_splits; ++k) {
    const int64_t waves = (base * k + nsm - 1) / nsm;
    const double cost = (double)waves * (4.0 + (double)nKt / (double)k);
    if (k == 1 || cost < best_cost) { best = k; best_cost = cost; }
  }
  p.Gp = gp;
  p.Rq = (int)rq;
  p.nQc = (int)nqc;
  p.splits = (int)best;
  return p;
}

int64_t split_ws_bytes(const lcattn_shape* s, const SplitPlan& p) {
  if (p.splits == 0) return 0;
  return align_up((int64_t)p.splits * s->B * s->Sq * s->Hq * s->D * 4, 256) +
         align_up((int64_t)p.splits * s->B * s->Hq * s->Sq * 4, 256);
}

}  // namespace

extern "C" {

size_t lcattn_fwd_workspace_size(const lcattn_shape* shape, const lcattn_mask_desc* mask) {
  lcattn_tile_meta_layout L;
  if (layout_of(shape, mask, &L) != LCATTN_OK) return 0;
  return (size_t)split_ws_bytes(shape, split_plan(shape, mask));
}

int lcattn_fwd_ws(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                  const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* o,
                  float* lse, void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  lcattn_tile_meta_layout L;
  int st = layout_of(shape, mask, &L);
  if (st) return st;
  const SplitPlan p = split_plan(shape, mask);
  if (p.splits == 0)
    return lcattn_fwd(shape, q, k, v, tile_meta, mask, scale, o, lse, stream);
  if (!q || !k || !v || !o || !lse || !tile_meta || !workspace) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(tile_meta) ||
      !aligned16(workspace))
    return LCATTN_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !(scale < 1e30f)) return LCATTN_ERR_INVALID_ARG;
  if ((int64_t)workspace_bytes < split_ws_bytes(shape, p)) return LCATTN_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv;
  if ((st = encode_bshd_box(&tq, q, shape->B, shape->Sq, shape->Hq, shape->D, shape->q_stride, p.Gp, p.Rq)))
    return st;
  if ((st = encode_bshd(&tk, k, shape->B, shape->Sk, shape->Hkv, shape->D, shape->k_stride))) return st;
  if ((st = encode_bshd(&tv, v, shape->B, shape->Sk, shape->Hkv, shape->D, shape->v_stride))) return st;
  SplitArgs a;
  a.pr = problem_of(shape);
  a.mask = mask_of(mask);
  a.meta = meta_of(L, tile_meta);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.Gp = p.Gp; a.Rq = p.Rq; a.nQc = p.nQc; a.splits = p.splits;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o_part = reinterpret_cast<float*>(ws);
  a.lse_part = reinterpret_cast<float*>(
      ws + align_up((int64_t)p.splits * shape->B * shape->Sq * shape->Hq * shape->D * 4, 256));
  a.o = o;
  a.o_sb = shape->o_stride[0]; a.o_ss = shape->o_stride[1]; a.o_sh = shape->o_stride[2];
  a.lse = lse;
  return cuda_status(launch_fwd_split(tq, tk, tv, a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Split partials of the e4m3 forward for a column-bounds mask (the only kind
// the split-KV path takes): the most any mask of this shape needs.
int64_t fwd8_split_bytes_max(const lcattn_shape* s) {
  lcattn_mask_desc cb{};
  cb.kind = LCATTN_MASK_COLBOUNDS;
  return split_ws_bytes(s, split_plan(s, &cb));
}

// The e4m3 forward on V^T already in device memory (vt: [B][Hkv][128][Skp]).
// Short query sides go through the split-KV kernel (partials in `workspace`),
// the rest through the persistent kernel (no workspace).
int fwd8_run(const lcattn_shape* shape, const void* q, const void* k, const void* vt, float q_scale,
             float k_scale, float v_scale, const void* tile_meta, const lcattn_mask_desc* mask, float scale,
             void* o, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t cs) {
  lcattn_tile_meta_layout L;
  int st = layout_of(shape, mask, &L);
  if (st) return st;
  if ((st = validate_fp8(shape))) return st;
  if (!q || !k || !vt || !o || !lse || !tile_meta) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned16(tile_meta))
    return LCATTN_ERR_UNSUPPORTED;
  for (float x : {scale, q_scale, k_scale, v_scale})
    if (!(x > 0.f) || !(x < 1e30f)) return LCATTN_ERR_INVALID_ARG;
  const int64_t skp = fp8_skp(shape);
  CUtensorMap tk, tvt;
  if ((st = encode_bshd8(&tk, k, shape->B, shape->Sk, shape->Hkv, shape->k_stride))) return st;
  if ((st = encode_vt8(&tvt, vt, shape->B, shape->Hkv, skp))) return st;
  const SplitPlan p = split_plan(shape, mask);
  if (p.splits > 0) {
    if (!workspace || !aligned16(workspace)) return LCATTN_ERR_INVALID_ARG;
    if ((int64_t)workspace_bytes < split_ws_bytes(shape, p)) return LCATTN_ERR_WORKSPACE;
    CUtensorMap tq;
    if ((st = encode_bshd8(&tq, q, shape->B, shape->Sq, shape->Hq, shape->q_stride, p.Gp, p.Rq))) return st;
    SplitArgs a;
    a.pr = problem_of(shape);
    a.mask = mask_of(mask);
    a.meta = meta_of(L, tile_meta);
    a.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
    a.o_scale = v_scale;
    a.Gp = p.Gp; a.Rq = p.Rq; a.nQc = p.nQc; a.splits = p.splits;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.o_part = reinterpret_cast<float*>(ws);
    a.lse_part = reinterpret_cast<float*>(
        ws + align_up((int64_t)p.splits * shape->B * shape->Sq * shape->Hq * shape->D * 4, 256));
    a.o = o;
    a.o_sb = shape->o_stride[0]; a.o_ss = shape->o_stride[1]; a.o_sh = shape->o_stride[2];
    a.lse = lse;
    return cuda_status(launch_fwd_split_e4m3(tq, tk, tvt, a, cs));
  }
  CUtensorMap tq, to;
  if ((st = encode_bshd8(&tq, q, shape->B, shape->Sq, shape->Hq, shape->q_stride))) return st;
  if ((st = encode_bshd(&to, o, shape->B, shape->Sq, shape->Hq, shape->D, shape->o_stride))) return st;
  FwdArgs a;
  a.pr = problem_of(shape);
  a.mask = mask_of(mask);
  a.meta = meta_of(L, tile_meta);
  a.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  a.o_scale = v_scale;
  a.o = o;
  a.o_sb = shape->o_stride[0]; a.o_ss = shape->o_stride[1]; a.o_sh = shape->o_stride[2];
  a.lse = lse;
  return cuda_status(launch_fwd_e4m3(tq, tk, tvt, to, a, cs));
}

}  // namespace

extern "C" {

size_t lcattn_fp8_vt_size(const lcattn_shape* shape) {
  if (validate_shape(shape) != LCATTN_OK || validate_fp8(shape) != LCATTN_OK) return 0;
  return (size_t)fwd8_ws_bytes(shape);
}

int lcattn_fp8_transpose_v(const lcattn_shape* shape, const void* v, void* vt, lcattn_stream_t stream) {
  int st = validate_shape(shape);
  if (st) return st;
  if ((st = validate_fp8(shape))) return st;
  if (!v || !vt) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(vt)) return LCATTN_ERR_UNSUPPORTED;
  return cuda_status(launch_vt8(static_cast<const uint8_t*>(v), shape->v_stride[0], shape->v_stride[1],
                                shape->v_stride[2], static_cast<uint8_t*>(vt), (int)shape->B, (int)shape->Sk,
                                (int)fp8_skp(shape), (int)shape->Hkv, reinterpret_cast<cudaStream_t>(stream)));
}

size_t lcattn_fwd_fp8_vt_workspace_size(const lcattn_shape* shape, const lcattn_mask_desc* mask) {
  lcattn_tile_meta_layout L;
  if (layout_of(shape, mask, &L) != LCATTN_OK || validate_fp8(shape) != LCATTN_OK) return 0;
  return (size_t)split_ws_bytes(shape, split_plan(shape, mask));
}

int lcattn_fwd_fp8_vt(const lcattn_shape* shape, const void* q, const void* k, const void* vt, float q_scale,
                      float k_scale, float v_scale, const void* tile_meta, const lcattn_mask_desc* mask, float scale,
                      void* o, float* lse, void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  return fwd8_run(shape, q, k, vt, q_scale, k_scale, v_scale, tile_meta, mask, scale, o, lse, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t lcattn_fwd_fp8_workspace_size(const lcattn_shape* shape) {
  if (validate_shape(shape) != LCATTN_OK || validate_fp8(shape) != LCATTN_OK) return 0;
  return (size_t)(fwd8_ws_bytes(shape) + fwd8_split_bytes_max(shape));
}

int lcattn_fwd_fp8(const lcattn_shape* shape, const void* q, const void* k, const void* v, float q_scale,
                   float k_scale, float v_scale, const void* tile_meta, const lcattn_mask_desc* mask, float scale,
                   void* o, float* lse, void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  lcattn_tile_meta_layout L;
  int st = layout_of(shape, mask, &L);
  if (st) return st;
  if ((st = validate_fp8(shape))) return st;
  if (!v || !workspace) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(workspace)) return LCATTN_ERR_UNSUPPORTED;
  // Workspace: V^T first, then the split partials (when the shape takes the split path).
  const int64_t vt_bytes = fwd8_ws_bytes(shape);
  const int64_t split_bytes = split_ws_bytes(shape, split_plan(shape, mask));
  if ((int64_t)workspace_bytes < vt_bytes + split_bytes) return LCATTN_ERR_WORKSPACE;
  for (float x : {scale, q_scale, k_scale, v_scale})
    if (!(x > 0.f) || !(x < 1e30f)) return LCATTN_ERR_INVALID_ARG;
  if (!q || !k || !o || !lse || !tile_meta) return LCATTN_ERR_INVALID_ARG;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if ((st = lcattn_fp8_transpose_v(shape, v, ws, stream))) return st;
  return fwd8_run(shape, q, k, ws, q_scale, k_scale, v_scale, tile_meta, mask, scale, o, lse,
                  split_bytes > 0 ? ws + vt_bytes : nullptr, (size_t)split_bytes, cs);
}

size_t lcattn_bwd_workspace_size(const lcattn_shape* shape) {
  if (validate_shape(shape) != LCATTN_OK) return 0;
  return (size_t)bwd_ws_bytes(shape, bwd_parts(shape), true);
}

}  // extern "C"

namespace {

// Caller-owned fp32 accumulators of the accumulate mode (all null otherwise).
struct AccumOut {
  float* dq = nullptr;
  float* dk = nullptr;
  float* dv = nullptr;
  bool on() const { return dq != nullptr; }
};

// Stages: bit 0 = pre-pass, bit 1 = dK/dV, bit 2 = dQ conversion.
int bwd_run(unsigned stages, const lcattn_shape* shape, const void* q, const void* k,
            const void* v, const void* o, const void* d_o, const float* lse,
            const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* dq, void* dk,
            void* dv, void* workspace, size_t workspace_bytes, lcattn_stream_t stream,
            bool allow_split = true, AccumOut acc = AccumOut(), bool deterministic = false) {
  lcattn_tile_meta_layout L;
  int st = layout_of(shape, mask, &L);
  if (st) return st;
  if (shape->D > 128 && deterministic) return LCATTN_ERR_UNSUPPORTED;  // no dQ kernel at head dim 256
  if (acc.on()) {
    if (!acc.dk || !acc.dv) return LCATTN_ERR_INVALID_ARG;
    // The outputs are the accumulators; the bf16 pointers are not used.
    dq = acc.dq; dk = acc.dk; dv = acc.dv;
  }
  if (!q || !k || !v || !o || !d_o || !lse || !tile_meta || !dq || !dk || !dv || !workspace)
    return LCATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, d_o, dq, dk, dv, workspace, tile_meta};
  for (auto p : ptrs)
    if (!aligned16(p)) return LCATTN_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !(scale < 1e30f)) return LCATTN_ERR_INVALID_ARG;
  // (The accumulate mode serves shards of a split sequence and never chunks;
  // the deterministic backward never chunks either: chunked units reduce-add.)
  const int64_t nchunks = allow_split && !acc.on() && !deterministic ? bwd_chunks(shape, mask) : 1;
  const int parts = allow_split ? bwd_parts(shape, nchunks) : 1;
  // Accumulate mode needs only D: dQ goes to the caller's accumulator and the
  // split units reduce-add their dK/dV shares directly.
  const int64_t need = acc.on() ? align_up(4 * shape->B * shape->Hq * shape->Sq, 256)
                     : deterministic ? bwd_det_ws_bytes(shape, parts)
                                     : bwd_ws_bytes(shape, nchunks > 1 ? 1 : parts, nchunks > 1);
  if ((int64_t)workspace_bytes < need) return LCATTN_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv, tdo;
  if ((st = encode_bshd(&tq, q, shape->B, shape->Sq, shape->Hq, shape->D, shape->q_stride))) return st;
  if ((st = encode_bshd(&tk, k, shape->B, shape->Sk, shape->Hkv, shape->D, shape->k_stride))) return st;
  if ((st = encode_bshd(&tv, v, shape->B, shape->Sk, shape->Hkv, shape->D, shape->v_stride))) return st;
  if ((st = encode_bshd(&tdo, d_o, shape->B, shape->Sq, shape->Hq, shape->D, shape->o_stride))) return st;
  BwdArgs a;
  a.pr = problem_of(shape);
  a.mask = mask_of(mask);
  a.meta = meta_of(L, tile_meta);
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o = o;
  a.d_o = d_o;
  a.o_sb = shape->o_stride[0]; a.o_ss = shape->o_stride[1]; a.o_sh = shape->o_stride[2];
  a.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.dvec = reinterpret_cast<float*>(ws);
  a.dq_acc = reinterpret_cast<float*>(ws + align_up(4 * shape->B * shape->Hq * shape->Sq, 256));
  a.parts = parts;
  a.dkv_part = reinterpret_cast<float*>(ws + (deterministic ? align_up(4 * shape->B * shape->Hq * shape->Sq, 256)
                                                             : bwd_ws_bytes(shape, 1, false)));
  a.nchunks = (int)nchunks;
  a.chunk_tiles = (int)kChunkTiles;
  a.red_parts = nchunks > 1 ? 1 : (parts > 1 ? parts : 0);
  // dQ from its own kernel (dq.cu: no fp32 reductions, so every output is
  // reproducible bit for bit) in the deterministic backward.  The fused form
  // (dQ partials reduce-added by the dK/dV kernel) is faster on every measured
  // workload but one: the separate kernel recomputes S and dP, 7 GEMMs against
  // 5 (dense 8K: 1018 against 1153 TFLOP/s; 128K block map: 1073 against 1053).
  a.dq_sep = deterministic ? 1 : 0;
  // The workspace accumulator is head-major, [B][Hq][Sq][D]: the rows one
  // head's dK/dV units add into are contiguous, so the units in flight (which
  // mostly work on the same head) keep a compact set of lines in L2.  The
  // caller's accumulator of the accumulate mode is [B][Sq][Hq][D].
  a.dqa_sb = shape->Hq * shape->Sq * shape->D;
  a.dqa_sh = shape->Sq * shape->D;
  a.dqa_ss = shape->D;
  a.accum = acc.on() ? 1 : 0;
  a.dk_acc = acc.dk;
  a.dv_acc = acc.dv;
  if (!acc.on() && nchunks > 1) {  // chunked units: dV then dK, fp32, in the partial slot
    a.dv_acc = a.dkv_part;
    a.dk_acc = a.dkv_part + shape->B * shape->Sk * shape->Hkv * shape->D;
  }
  if (acc.on()) {
    a.dq_acc = acc.dq;
    a.dqa_sb = shape->Sq * shape->Hq * shape->D;
    a.dqa_ss = shape->Hq * shape->D;
    a.dqa_sh = shape->D;
    a.dkv_part = nullptr;
    stages &= 3u;  // no bf16 conversion: the accumulators are the outputs
  }
  a.dq = dq;
  a.q_sb = shape->q_stride[0]; a.q_ss = shape->q_stride[1]; a.q_sh = shape->q_stride[2];
  a.dk = dk;
  a.k_sb = shape->k_stride[0]; a.k_ss = shape->k_stride[1]; a.k_sh = shape->k_stride[2];
  a.dv = dv;
  a.v_sb = shape->v_stride[0]; a.v_ss = shape->v_stride[1]; a.v_sh = shape->v_stride[2];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (stages & 1u) e = launch_bwd_prepass(a, s);
  if (e == cudaSuccess && (stages & 2u)) e = launch_bwd_dkdv(tq, tk, tv, tdo, a, s);
  if (e == cudaSuccess && (stages & 4u))
    e = a.dq_sep ? launch_bwd_dq(tq, tk, tv, tdo, a, s) : launch_bwd_dq_convert(a, s);
  return cuda_status(e);
}

}  // namespace

extern "C" {

int lcattn_bwd(const lcattn_shape* shape, const void* q, const void* k, const void* v,
               const void* o, const void* d_o, const float* lse, const void* tile_meta,
               const lcattn_mask_desc* mask, float scale, void* dq, void* dk, void* dv,
               void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  return bwd_run(7u, shape, q, k, v, o, d_o, lse, tile_meta, mask, scale, dq, dk, dv, workspace,
                 workspace_bytes, stream);
}

int lcattn_bwd_stage(int stage, const lcattn_shape* shape, const void* q, const void* k,
                     const void* v, const void* o, const void* d_o, const float* lse,
                     const void* tile_meta, const lcattn_mask_desc* mask, float scale, void* dq,
                     void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     lcattn_stream_t stream) {
  if (stage < 1 || stage > 3) return LCATTN_ERR_INVALID_ARG;
  return bwd_run(1u << (stage - 1), shape, q, k, v, o, d_o, lse, tile_meta, mask, scale, dq, dk,
                 dv, workspace, workspace_bytes, stream);
}

size_t lcattn_bwd_deterministic_workspace_size(const lcattn_shape* shape) {
  if (validate_shape(shape) != LCATTN_OK || shape->D > 128) return 0;
  return (size_t)bwd_det_ws_bytes(shape, bwd_parts(shape));
}

int lcattn_bwd_deterministic(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                             const void* o, const void* d_o, const float* lse, const void* tile_meta,
                             const lcattn_mask_desc* mask, float scale, void* dq, void* dk, void* dv,
                             void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  return bwd_run(7u, shape, q, k, v, o, d_o, lse, tile_meta, mask, scale, dq, dk, dv, workspace,
                 workspace_bytes, stream, /*allow_split=*/true, AccumOut(), /*deterministic=*/true);
}

size_t lcattn_bwd_accum_workspace_size(const lcattn_shape* shape) {
  if (validate_shape(shape) != LCATTN_OK) return 0;
  return (size_t)align_up(4 * shape->B * shape->Hq * shape->Sq, 256);
}

int lcattn_bwd_accum(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                     const void* o, const void* d_o, const float* lse, const void* tile_meta,
                     const lcattn_mask_desc* mask, float scale, float* dq_acc, float* dk_acc,
                     float* dv_acc, void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  if (!dq_acc || !dk_acc || !dv_acc) return LCATTN_ERR_INVALID_ARG;
  AccumOut acc;
  acc.dq = dq_acc; acc.dk = dk_acc; acc.dv = dv_acc;
  return bwd_run(3u, shape, q, k, v, o, d_o, lse, tile_meta, mask, scale, nullptr, nullptr, nullptr,
                 workspace, workspace_bytes, stream, /*allow_split=*/true, acc);
}

int lcattn_mask_shard(const lcattn_mask_desc* global, int64_t B, int64_t Sq, int64_t Sk, int64_t q0,
                      int64_t Sq_s, int64_t k0, int64_t Sk_s, int32_t* col_bounds_out,
                      int32_t* row_bounds_out, int32_t* q_offs_out, int32_t* k_offs_out,
                      lcattn_stream_t stream) {
  if (!global || B < 1 || B > 65535 || Sq < 1 || Sk < 1 || Sq > kMaxSeq || Sk > kMaxSeq)
    return LCATTN_ERR_INVALID_ARG;
  if (q0 < 0 || Sq_s < 1 || q0 + Sq_s > Sq || k0 < 0 || Sk_s < 1 || k0 + Sk_s > Sk)
    return LCATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (global->kind == LCATTN_MASK_COLBOUNDS) {
    if (!global->col_bounds || !aligned16(global->col_bounds) || !col_bounds_out ||
        !aligned16(col_bounds_out))
      return LCATTN_ERR_INVALID_ARG;
    if (row_bounds_out && (!global->row_bounds || !aligned16(global->row_bounds) ||
                           !aligned16(row_bounds_out)))
      return LCATTN_ERR_INVALID_ARG;
    ShardBoundsArgs c;
    c.in = reinterpret_cast<const int4*>(global->col_bounds);
    c.out = reinterpret_cast<int4*>(col_bounds_out);
    c.S_in = Sk; c.start = k0; c.n = Sk_s; c.B = (int)B; c.shift = (int)q0; c.limit = (int)Sq_s;
    cudaError_t e = launch_shard_bounds(c, s);
    if (e == cudaSuccess && row_bounds_out) {
      ShardBoundsArgs r;
      r.in = reinterpret_cast<const int4*>(global->row_bounds);
      r.out = reinterpret_cast<int4*>(row_bounds_out);
      r.S_in = Sq; r.start = q0; r.n = Sq_s; r.B = (int)B; r.shift = (int)k0; r.limit = (int)Sk_s;
      e = launch_shard_bounds(r, s);
    }
    return cuda_status(e);
  }
  if (global->kind == LCATTN_MASK_BLOCKMAP) {
    if (!global->q_block_offs || !global->k_block_offs || !q_offs_out || !k_offs_out ||
        global->nQb < 1 || global->nKb < 1)
      return LCATTN_ERR_INVALID_ARG;
    cudaError_t e = launch_shard_offsets(global->q_block_offs, q_offs_out, global->nQb, (int)q0,
                                         (int)Sq_s, s);
    if (e == cudaSuccess)
      e = launch_shard_offsets(global->k_block_offs, k_offs_out, global->nKb, (int)k0, (int)Sk_s, s);
    return cuda_status(e);
  }
  return LCATTN_ERR_INVALID_ARG;
}

int lcattn_lse_merge(const lcattn_shape* shape, float* o_acc, float* lse_acc, const void* o_part,
                     const float* lse_part, void* o_out, const int64_t* o_out_stride, int first,
                     lcattn_stream_t stream) {
  int st = validate_shape(shape);
  if (st) return st;
  if (!o_acc || !lse_acc || !o_part || !lse_part) return LCATTN_ERR_INVALID_ARG;
  if (first != 0 && first != 1) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(o_acc) || !aligned16(o_part) || (o_out && !aligned16(o_out)) ||
      (reinterpret_cast<uintptr_t>(lse_acc) & 3u) || (reinterpret_cast<uintptr_t>(lse_part) & 3u))
    return LCATTN_ERR_UNSUPPORTED;
  MergeArgs a;
  a.pr = problem_of(shape);
  a.o_acc = o_acc; a.lse_acc = lse_acc;
  a.o_part = o_part;
  a.p_sb = shape->o_stride[0]; a.p_ss = shape->o_stride[1]; a.p_sh = shape->o_stride[2];
  a.lse_part = lse_part;
  a.o_out = o_out;
  const int64_t* os = o_out_stride ? o_out_stride : shape->o_stride;
  if (o_out) {
    for (int i = 0; i < 3; ++i) {
      if (os[i] < 0) return LCATTN_ERR_INVALID_ARG;
      if (os[i] % 8 != 0) return LCATTN_ERR_UNSUPPORTED;
    }
    if (os[2] < shape->D || os[1] < shape->D || (shape->B > 1 && os[0] < shape->D)) return LCATTN_ERR_INVALID_ARG;
  }
  a.o_sb = os[0]; a.o_ss = os[1]; a.o_sh = os[2];
  a.first = first;
  return cuda_status(launch_lse_merge(a, reinterpret_cast<cudaStream_t>(stream)));
}

int lcattn_f32_to_bf16(const float* src, void* dst, int64_t B, int64_t S, int64_t H, int64_t D,
                       const int64_t dst_stride[3], lcattn_stream_t stream) {
  if (!src || !dst || !dst_stride || B < 1 || S < 1 || H < 1) return LCATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return LCATTN_ERR_UNSUPPORTED;
  for (int i = 0; i < 3; ++i) {
    if (dst_stride[i] < 0) return LCATTN_ERR_INVALID_ARG;
    if (dst_stride[i] % 8 != 0) return LCATTN_ERR_UNSUPPORTED;
  }
  if (dst_stride[2] < D || dst_stride[1] < D || (B > 1 && dst_stride[0] < D)) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return LCATTN_ERR_UNSUPPORTED;
  return cuda_status(launch_f32_to_bf16(src, dst, B, S, H, D, dst_stride[0], dst_stride[1], dst_stride[2],
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Backward scratch (D vector + fp32 dQ accumulator) for lcattn_bwd_noalloc.
// In host code this name is only a stand-in for the device array; kernels get
// the device address that cudaGetSymbolAddress returns.
static __device__ __align__(256) uint8_t g_noalloc_scratch[LCATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LCATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LCATTN_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return LCATTN_OK;
}

}  // namespace

extern "C" {

int lcattn_bwd_noalloc(const lcattn_shape* shape, const void* q, const void* k, const void* v,
                       const void* o, const void* d_o, const float* lse, const void* tile_meta,
                       const lcattn_mask_desc* mask, float scale, void* dq, void* dk, void* dv,
                       lcattn_stream_t stream) {
  int st = validate_shape(shape);
  if (st) return st;
  // No split here: the fixed array holds D and the dQ accumulator only.
  const int64_t need = bwd_ws_bytes(shape, 1, false);
  if (need > (int64_t)LCATTN_NOALLOC_SCRATCH_BYTES) return LCATTN_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws))) return st;
  return bwd_run(7u, shape, q, k, v, o, d_o, lse, tile_meta, mask, scale, dq, dk, dv, ws,
                 (size_t)LCATTN_NOALLOC_SCRATCH_BYTES, stream, /*allow_split=*/false);
}

}  // extern "C"

namespace {

int validate_select(const lcattn_shape* s, const lcattn_select_desc* d) {
  int st = validate_shape(s);
  if (st) return st;
  if (!d || !d->q_block_offs || !d->k_block_offs) return LCATTN_ERR_INVALID_ARG;
  if (d->rule == LCATTN_SELECT_TOPK) {
    if (d->top_k < 0) return LCATTN_ERR_INVALID_ARG;
  } else if (d->rule == LCATTN_SELECT_TOPP) {
    if (!(d->top_p == d->top_p) || d->top_p > 3.0e38f || d->top_p < -3.0e38f)
      return LCATTN_ERR_INVALID_ARG;  // NaN or infinite
  } else {
    return LCATTN_ERR_INVALID_ARG;
  }
  if (d->causal != 0 && d->causal != 1) return LCATTN_ERR_INVALID_ARG;
  if (d->nQb < 1 || d->nKb < 1 || d->nQb > s->Sq || d->nKb > s->Sk) return LCATTN_ERR_INVALID_ARG;
  if (d->nKb > LCATTN_SELECT_MAX_KB) return LCATTN_ERR_UNSUPPORTED;
  if (s->D != 128) return LCATTN_ERR_UNSUPPORTED;  // block means are taken over 128 columns
  // Grid sizes of the two kernels.
  const int64_t slabs_q = (s->Hq + 7) / 8, slabs_k = (s->Hkv + 7) / 8;
  if (s->B * (d->nQb * slabs_q + d->nKb * slabs_k) >= (int64_t(1) << 31)) return LCATTN_ERR_UNSUPPORTED;
  if (s->B * s->Hq * (int64_t)d->nQb >= (int64_t(1) << 31)) return LCATTN_ERR_UNSUPPORTED;
  return LCATTN_OK;
}

int64_t select_ws_bytes(const lcattn_shape* s, const lcattn_select_desc* d) {
  return align_up(4 * kD * s->B * s->Hq * (int64_t)d->nQb, 256) +
         align_up(4 * kD * s->B * s->Hkv * (int64_t)d->nKb, 256);
}

int select_run(unsigned stages, const lcattn_shape* shape, const void* q, const void* k,
               const lcattn_select_desc* sel, float scale, uint8_t* block_map, float* scores,
               void* workspace, size_t workspace_bytes, lcattn_stream_t stream) {
  int st = validate_select(shape, sel);
  if (st) return st;
  if (!q || !k || !block_map || !workspace) return LCATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(workspace)) return LCATTN_ERR_UNSUPPORTED;
  if (scores && (reinterpret_cast<uintptr_t>(scores) & 3u)) return LCATTN_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !(scale < 1e30f)) return LCATTN_ERR_INVALID_ARG;
  if ((int64_t)workspace_bytes < select_ws_bytes(shape, sel)) return LCATTN_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* qbar = reinterpret_cast<float*>(ws);
  float* kbar = reinterpret_cast<float*>(ws + align_up(4 * kD * shape->B * shape->Hq * (int64_t)sel->nQb, 256));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (stages & 1u) {
    PoolSide qs, ks;
    qs.x = static_cast<const uint16_t*>(q);
    qs.sb = shape->q_stride[0]; qs.ss = shape->q_stride[1]; qs.sh = shape->q_stride[2];
    qs.B = (int)shape->B; qs.S = (int)shape->Sq; qs.H = (int)shape->Hq; qs.nb = sel->nQb;
    qs.slabs = (int)((shape->Hq + 7) / 8); qs.offs = sel->q_block_offs; qs.out = qbar;
    qs.transposed = 0;
    ks.x = static_cast<const uint16_t*>(k);
    ks.sb = shape->k_stride[0]; ks.ss = shape->k_stride[1]; ks.sh = shape->k_stride[2];
    ks.B = (int)shape->B; ks.S = (int)shape->Sk; ks.H = (int)shape->Hkv; ks.nb = sel->nKb;
    ks.slabs = (int)((shape->Hkv + 7) / 8); ks.offs = sel->k_block_offs; ks.out = kbar;
    ks.transposed = 1;
    e = launch_block_pool(qs, ks, s);
  }
  if (e == cudaSuccess && (stages & 2u)) {
    SelectArgs a;
    a.qbar = qbar; a.kbar = kbar;
    a.q_offs = sel->q_block_offs; a.k_offs = sel->k_block_offs;
    a.B = (int)shape->B; a.Hq = (int)shape->Hq; a.G = (int)(shape->Hq / shape->Hkv);
    a.nQb = sel->nQb; a.nKb = sel->nKb; a.Sq = (int)shape->Sq; a.Sk = (int)shape->Sk;
    a.rule = sel->rule; a.top_k = sel->top_k; a.top_p = sel->top_p; a.causal = sel->causal;
    a.scale = scale; a.map = block_map; a.scores = scores;
    select_geometry(sel->nKb, &a.R, &a.n2);
    e = launch_block_select(a, s);
  }
  return cuda_status(e);
}

}  // namespace

extern "C" {

size_t lcattn_block_select_workspace_size(const lcattn_shape* shape, const lcattn_select_desc* sel) {
  if (validate_select(shape, sel) != LCATTN_OK) return 0;
  return (size_t)select_ws_bytes(shape, sel);
}

int lcattn_block_select(const lcattn_shape* shape, const void* q, const void* k,
                        const lcattn_select_desc* sel, float scale, uint8_t* block_map,
                        float* scores, void* workspace, size_t workspace_bytes,
                        lcattn_stream_t stream) {
  return select_run(3u, shape, q, k, sel, scale, block_map, scores, workspace, workspace_bytes,
                    stream);
}

int lcattn_block_select_stage(int stage, const lcattn_shape* shape, const void* q, const void* k,
                              const lcattn_select_desc* sel, float scale, uint8_t* block_map,
                              float* scores, void* workspace, size_t workspace_bytes,
                              lcattn_stream_t stream) {
  if (stage < 1 || stage > 2) return LCATTN_ERR_INVALID_ARG;
  return select_run(1u << (stage - 1), shape, q, k, sel, scale, block_map, scores, workspace,
                    workspace_bytes, stream);
}

int lcattn_read_status(const void* tile_meta, lcattn_stream_t stream) {
  if (!tile_meta) return LCATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return LCATTN_ERR_CUDA;
  int32_t w[4] = {0, 0, 0, 0};
  if (cudaMemcpy(w, tile_meta, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LCATTN_ERR_CUDA;
  for (int i = 0; i < 4; ++i)
    if (w[i] != 0) return w[i];
  return LCATTN_OK;
}

int lcattn_selftest_wait_timeout(void* tile_meta, lcattn_stream_t stream) {
  if (!tile_meta || !aligned16(tile_meta)) return LCATTN_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait_timeout(static_cast<int32_t*>(tile_meta),
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

int lcattn_clear_status(void* tile_meta, lcattn_stream_t stream) {
  if (!tile_meta) return LCATTN_ERR_INVALID_ARG;
  // Status words and the scheduler words behind them (offsets 0 and 16 for every layout).
  return cuda_status(cudaMemsetAsync(tile_meta, 0, 32, reinterpret_cast<cudaStream_t>(stream)));
}

const char* lcattn_status_string(int status) {
  switch (status) {
    case LCATTN_OK: return "ok";
    case LCATTN_ERR_INVALID_ARG: return "invalid argument";
    case LCATTN_ERR_UNSUPPORTED: return "unsupported shape, stride, alignment or head dim";
    case LCATTN_ERR_WORKSPACE: return "buffer smaller than required";
    case LCATTN_ERR_CUDA: return "CUDA error";
    case LCATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting (bounded device wait expired)";
    case LCATTN_ERR_DEVICE_MASK: return "block offsets are not nondecreasing from 0 to the sequence length";
    case LCATTN_ERR_SCRATCH_LIMIT:
      return "problem needs more backward scratch than the fixed no-allocation array holds";
    default: return "unknown status";
  }
}

int lcattn_version(void) { return 100; }

}  // extern "C"
