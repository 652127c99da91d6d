// Internal declarations shared by the host layer (api.cu) and the kernel
// translation units.  Nothing here is part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/lcattn.h"

namespace lcattn {

constexpr int kBM = LCATTN_BLOCK_M;  // query rows per tile
constexpr int kBN = LCATTN_BLOCK_N;  // key columns per tile
constexpr int kD = 128;              // head dim

// Mask descriptor as the kernels see it.
struct MaskDev {
  int kind;                  // LCATTN_MASK_COLBOUNDS / LCATTN_MASK_BLOCKMAP
  const int4* col_bounds;    // [B][Sk] {a0,b0,a1,b1}
  const int4* row_bounds;    // [B][Sq] {c0,d0,c1,d1}, or null (column bounds only)
  const uint8_t* block_map;  // [B][Hq][nQb][nKb]
  const int32_t* q_offs;     // [nQb+1]
  const int32_t* k_offs;     // [nKb+1]
  int nQb, nKb;
};

// Pointers into a tile-meta buffer.
struct TileMetaDev {
  int32_t* status;
  unsigned long long* sched;  // [0] next forward item, [1] forward CTAs done fetching
  uint8_t* cls;
  int32_t* fwd_cnt;
  int32_t* fwd_lst;
  int32_t* fwd_ord;
  int32_t* bwd_cnt;
  int32_t* bwd_lst;
  int32_t* bwd_ord;
  int nQt, nKt, nH, B;
};

struct ProblemDev {
  int B, Sq, Sk, Hq, Hkv, G;
  int D;  // head dim: 64 or 128
};

// ---- launchers (defined in the kernel translation units) -----------------
cudaError_t launch_mask_compile(const ProblemDev& pr, const MaskDev& m, const TileMetaDev& t,
                                cudaStream_t st);

struct FwdArgs {
  ProblemDev pr;
  MaskDev mask;
  TileMetaDev meta;
  float scale_log2;         // scale * log2(e) (e4m3: times the Q and K factors)
  float o_scale = 1.f;      // factor of O / l (e4m3: the V factor)
  void* o;
  int64_t o_sb, o_ss, o_sh;
  float* lse;
};
// `to`: O as a TMA map with the same box as Q (the epilogue's stores).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& a, cudaStream_t st);
// The same forward with e4m3 Q and K (maps of 128-byte boxes) and `tvt`
// mapping V^T [B][Hkv][128][Skp] e4m3 (box: 128 keys x 128 head-dim rows);
// D = 128, O bf16.  a.scale_log2 carries the Q and K factors, a.o_scale the V factor.
cudaError_t launch_fwd_e4m3(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                            const CUtensorMap& to, const FwdArgs& a, cudaStream_t st);

// Split-KV forward for short query sides (fwd_split.cu).
struct SplitArgs {
  ProblemDev pr;
  MaskDev mask;             // column bounds (+ optional row bounds) only
  TileMetaDev meta;
  float scale_log2;
  int Gp;                   // query heads packed per tile (a power of two dividing G)
  int Rq;                   // query positions per tile, Gp * Rq = 128
  int nQc;                  // query chunks, ceil(Sq / Rq)
  int splits;               // slices of each key-tile list
  float o_scale = 1.f;      // factor of O / l (e4m3: the V factor)
  float* o_part;            // [splits][B][Sq][Hq][128] fp32, O / l of each slice
  float* lse_part;          // [splits][B][Hq][Sq]
  void* o;
  int64_t o_sb, o_ss, o_sh;
  float* lse;
};
int split_heads_packed(int G);
cudaError_t launch_fwd_split(const CUtensorMap& tq_packed, const CUtensorMap& tk,
                             const CUtensorMap& tv, const SplitArgs& a, cudaStream_t st);
// The same with e4m3 Q (packed box of 128 bytes x Gp heads x Rq rows) and K,
// and `tvt` mapping V^T [B][Hkv][128][Skp] e4m3; a.scale_log2 carries the Q and
// K factors, a.o_scale the V factor.  D = 128.
cudaError_t launch_fwd_split_e4m3(const CUtensorMap& tq_packed, const CUtensorMap& tk, const CUtensorMap& tvt,
                                  const SplitArgs& a, cudaStream_t st);

struct BwdArgs {
  ProblemDev pr;
  MaskDev mask;
  TileMetaDev meta;
  float scale;
  float scale_log2;
  const void* o;
  const void* d_o;
  int64_t o_sb, o_ss, o_sh;
  const float* lse;
  float* dvec;   // D [B][Hq][Sq]
  float* dq_acc; // fp32 dQ accumulator, element strides below (head dim contiguous)
  int64_t dqa_sb, dqa_ss, dqa_sh;
  int parts;       // dK/dV units split over this many shares of the GQA group's heads (1: none)
  float* dkv_part; // parts > 1: fp32 partials [parts][dV, dK][B][Sk][Hkv][128]
  // Accumulate mode (context-parallel shards): dq_acc is the caller's fp32
  // accumulator and is not zeroed; dK and dV are reduce-added in fp32 into
  // dk_acc / dv_acc [B][Sk][Hkv][D] instead of being stored as bf16.
  int accum;
  float* dk_acc;
  float* dv_acc;
  // Chunked units (per-head lists): each (key tile, KV head) unit is split
  // into nchunks units over query-tile ranges of chunk_tiles tiles; their dK
  // and dV go into the fp32 accumulator at dkv_part ([dV, dK][B][Sk][Hkv][D]).
  int nchunks, chunk_tiles;
  // fp32 dK/dV slots the reduction kernel sums into the bf16 outputs (0 = none).
  int red_parts;
  // 1: dQ from the separate dQ kernel (dq.cu), written as bf16 with no fp32
  // accumulator; the dK/dV kernel then skips its dQ product.
  int dq_sep;
  void* dq;
  int64_t q_sb, q_ss, q_sh;
  void* dk;
  int64_t k_sb, k_ss, k_sh;
  void* dv;
  int64_t v_sb, v_ss, v_sh;
};
cudaError_t launch_bwd_prepass(const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_dq_convert(const BwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st);

// ---- FP8 forward: the V^T pre-pass (fwd8.cu) ---------------------------------
// V [B][Sk][Hkv][128] e4m3 (byte strides) -> V^T [B][Hkv][128][Skp] e4m3, keys
// in [Sk, Skp) written as 0.  The forward is launch_fwd_e4m3 (fwd.cu).
cudaError_t launch_vt8(const uint8_t* v, int64_t v_sb, int64_t v_ss, int64_t v_sh, uint8_t* vt, int B, int Sk,
                       int Skp, int Hkv, cudaStream_t st);

// ---- context-parallel building blocks (ring.cu) ---------------------------
// Column / row bounds of one shard pair: out = clamp(in - shift, 0, limit),
// per int32, over n int4 entries of each batch's window [start, start + n).
struct ShardBoundsArgs {
  const int4* in;      // [B][S_in] global bounds
  int4* out;           // [B][n]
  int64_t S_in, start, n;
  int B;
  int shift, limit;
};
cudaError_t launch_shard_bounds(const ShardBoundsArgs& a, cudaStream_t st);
// Block offsets of one shard: out[i] = clamp(in[i] - shift, 0, limit), i <= n.
cudaError_t launch_shard_offsets(const int32_t* in, int32_t* out, int n, int shift, int limit,
                                 cudaStream_t st);

struct MergeArgs {
  ProblemDev pr;
  float* o_acc;         // [B][Sq][Hq][D] fp32
  float* lse_acc;       // [B][Hq][Sq]
  const void* o_part;   // bf16 with o_part strides
  int64_t p_sb, p_ss, p_sh;
  const float* lse_part;
  void* o_out;          // bf16 with o_out strides, or null
  int64_t o_sb, o_ss, o_sh;
  int first;
};
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t st);

// fp32 [B][S][H][D] contiguous -> bf16 with strides (b, s, h).
cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t B, int64_t S, int64_t H, int64_t D,
                               int64_t sb, int64_t ss, int64_t sh, cudaStream_t st);
cudaError_t launch_selftest_wait_timeout(int32_t* status, cudaStream_t st);

// ---- dynamic block selection (select.cu) ---------------------------------
// One side (Q or K) of the block-mean pass.
struct PoolSide {
  const uint16_t* x;        // bf16 [B][S][H][128], element strides below
  int64_t sb, ss, sh;
  int B, S, H, nb, slabs;   // slabs = ceil(H / 8)
  const int32_t* offs;      // [nb + 1], read clamped to [0, S]
  float* out;               // block means, [B][H][nb][128] or (transposed) [B][H][128][nb]
  int transposed;
};
cudaError_t launch_block_pool(const PoolSide& qs, const PoolSide& ks, cudaStream_t st);

struct SelectArgs {
  const float* qbar;        // [B][Hq][nQb][128]
  const float* kbar;        // [B][Hkv][128][nKb]
  const int32_t* q_offs;
  const int32_t* k_offs;
  int B, Hq, G, nQb, nKb, Sq, Sk;
  int rule, top_k;
  float top_p;
  int causal;
  float scale;
  uint8_t* map;             // [B][Hq][nQb][nKb]
  float* scores;            // same shape, or null
  int R, n2;                // query blocks per CTA; sort width (power of two >= nKb, >= 32)
};
void select_geometry(int nKb, int* R, int* n2);
size_t select_smem_bytes(int R, int n2, int nKb);
cudaError_t launch_block_select(const SelectArgs& a, cudaStream_t st);

}  // namespace lcattn
