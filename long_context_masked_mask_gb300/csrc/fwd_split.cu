// Split-KV forward for short query sides: decode-style rows and short query
// chunks against a long key sequence (query and key lengths that differ,
// bottom-right aligned; the variants the pages' kernels take, xllm-io blog
// review, sections "密集注意力内核" and "稀疏注意力内核").
//
// With few query rows the regular forward has too few work items to fill the
// GPU, and each item walks the whole key list alone.  Here:
//   * the query heads of a GQA group that read the same K/V are packed into one
//     128-row tile: row r is query position r / Gp of head r % Gp (Gp heads x
//     Rq positions, Gp * Rq = 128), loaded by one TMA box of Gp heads x Rq rows,
//     so each K/V tile is read once per group instead of once per head pair;
//   * the key-tile list of every (batch, KV group, query chunk) is split into
//     `splits` contiguous slices, one CTA per slice, each writing O / l (fp32)
//     and its LSE to a workspace;
//   * combine_kernel merges the slices: LSE = log sum_c exp(LSE_c),
//     O = sum_c exp(LSE_c - LSE) O_c, written as bf16 with the final LSE.
// The per-tile pipeline is the regular forward's one-head mode: a K/V ring (4
// stages of 128-wide tiles, 8 of 64-wide ones), S double-buffered in TMEM and
// issued one tile ahead of PV, P written
// over S as bf16 and read from TMEM by the PV GEMM.  Column-bounds masks only
// (the packed rows of different heads share the mask).
// The same kernel runs e4m3 Q and K with V^T tiles (F8): kind::f8f6f4
// products, P as e4m3(16 P) under a rescale threshold of 4 -- the arithmetic
// of the persistent forward's e4m3 instantiation.
#include <cuda_bf16.h>

#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

using namespace dev;

// Head dim D (64, 128 or 256): tiles are 128 rows x D bf16 (D/64 boxes of 64
// columns); the K/V ring holds 128 KB.  A ring entry is a whole K or V tile for
// D <= 128 (8 or 4 stages) and a head-dim half of one at D = 256 (4 stages of
// 32 KB, so the next tile's K streams in while this tile is consumed).
// F8 (e4m3, D = 128): a tile is 128 rows x 128 bytes, one box; the V entries
// are V^T tiles (keys contiguous), 8 stages of 16 KB.
template <int D, bool F8 = false> struct SplitGeom {
  static_assert(!F8 || D == 128, "the e4m3 path is built for head dim 128");
  static constexpr int kElem = F8 ? 1 : 2;
  static constexpr int kTileBytes = 128 * D * kElem;
  static constexpr int kBoxCols = F8 ? 128 : 64;   // elements per 128-byte box row
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kParts = D == 256 ? 2 : 1;
  static constexpr int kEntryBytes = kTileBytes / kParts;
  static constexpr int kBoxesPerEntry = kBoxes / kParts;
  static constexpr int kStages = (D == 64 || F8) ? 8 : 4;
  static constexpr int kSSteps = D * kElem / 32 / kParts;  // S k-steps of 32 bytes per entry
  static constexpr int kPvSteps = F8 ? 4 : 8;              // PV k-steps (8 TMEM columns of P each)
  static constexpr float kRescaleThreshold = F8 ? 4.0f : 8.0f;
  static constexpr float kLog2PScale = F8 ? 4.0f : 0.0f;   // e4m3 P is stored as P * 2^4
};
constexpr int kHalfBytes = 16384;
constexpr int kThreads = 256;  // warps 0-3 softmax, 4 producer, 5 MMA, 6-7 idle

template <int D, bool F8 = false>
struct SplitSmem {
  static constexpr int kStages = SplitGeom<D, F8>::kStages;
  static constexpr int kTileBytes = SplitGeom<D, F8>::kTileBytes;
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t kv[kStages][SplitGeom<D, F8>::kEntryBytes];
  int4 bnd[2][kBN];
  uint64_t bnd_ready[2];
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full;   // one phase per PV
  uint64_t o_done;   // the slice's last PV has completed
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int base) {
  const int a = max(lo, base), b = min(hi, base + 32);
  if (b <= a) return 0u;
  const int n = b - a;
  return (n == 32) ? 0xffffffffu : (((1u << n) - 1u) << (a - base));
}

struct Unit {
  int b, g, hs, qc, c;
};

__device__ __forceinline__ Unit unit_of(const SplitArgs& a, int u) {
  Unit x;
  const int nhs = a.pr.G / a.Gp;
  x.hs = u % nhs; u /= nhs;
  x.c = u % a.splits; u /= a.splits;
  x.qc = u % a.nQc; u /= a.nQc;
  x.g = u % a.pr.Hkv;
  x.b = u / a.pr.Hkv;
  return x;
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
split_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ SplitArgs a) {
  constexpr int kStages = SplitGeom<D, F8>::kStages;
  constexpr int kTileBytes = SplitGeom<D, F8>::kTileBytes;
  constexpr int kBoxes = SplitGeom<D, F8>::kBoxes;
  constexpr int kParts = SplitGeom<D, F8>::kParts;
  constexpr int kEntryBytes = SplitGeom<D, F8>::kEntryBytes;
  constexpr int kBoxesPerEntry = SplitGeom<D, F8>::kBoxesPerEntry;
  constexpr int kBoxCols = SplitGeom<D, F8>::kBoxCols;
  constexpr int kE = 2 * kParts;  // ring entries per key tile
  // Half-tile entries: K runs a tile ahead of V (K(0), K(1), V(0), ..., V(n-1)),
  // the order the MMA warp consumes them.
  constexpr bool kAhead = kParts == 2;
  extern __shared__ uint8_t smem_raw[];
  SplitSmem<D, F8>& sm = *reinterpret_cast<SplitSmem<D, F8>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const ProblemDev& pr = a.pr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* gstatus = a.meta.status;
  const Unit un = unit_of(a, blockIdx.x);
  const int qs0 = un.qc * a.Rq;                // first query position of the tile
  const int qt = qs0 / kBM;                     // the mask compiler's query tile holding it
  const int64_t lbase = (int64_t)un.b * a.meta.nQt;  // column bounds: one list per batch entry
  const int n_all = __ldg(a.meta.fwd_cnt + lbase + qt);
  const int j_lo = (int)(((int64_t)n_all * un.c) / a.splits);
  const int j_hi = (int)(((int64_t)n_all * (un.c + 1)) / a.splits);
  const int n = j_hi - j_lo;
  const int32_t* list = a.meta.fwd_lst + (lbase + qt) * a.meta.nKt + j_lo;
  const int h_first = un.g * pr.G + un.hs * a.Gp;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], 128);
      mbar_init(&sm.bnd_ready[s], 128);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 4 && n > 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    bool ok = true;
    int t = 0;
    auto load_entry = [&](const CUtensorMap* tm, int kt, int part) -> bool {
      const int stage = t % kStages, use = t / kStages;
      if (use > 0) {
        const bool okw = mbar_wait(&sm.kv_empty[stage], (use - 1) & 1, abort_flag, gstatus,
                                   LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, okw)) return false;
      }
      mbar_expect_tx_e(&sm.kv_full[stage], kEntryBytes);
      if (F8 && tm == &tmV) {
        // V^T [B][Hkv][128][keys]: the 128 keys of tile kt x all 128 head-dim rows.
        tma_load_4d_e(sm.kv[stage], tm, &sm.kv_full[stage], kt * kBN, 0, un.g, un.b);
      } else {
        for (int bx = 0; bx < kBoxesPerEntry; ++bx)
          tma_load_4d_e(sm.kv[stage] + bx * kHalfBytes, tm, &sm.kv_full[stage], 128 * part + kBoxCols * bx,
                        un.g, kt * kBN, un.b);
      }
      ++t;
      return true;
    };
    for (int u = 0; u < kE * n; ++u) {
      const int j = u / kE, e = u % kE;
      const int part = e % kParts;
      const bool is_v = e >= kParts;
      if (!(kAhead && is_v && j == 0)) {  // K ahead of V: no V before the first K pair
        const int kt = __ldg(list + (kAhead && is_v ? j - 1 : j)) >> 1;
        if (!load_entry(is_v ? &tmV : &tmK, kt, part)) { ok = false; break; }
      }
      if (u == 0) {
        // Packed query tile: Gp heads x Rq positions; row = position * Gp + head.
        mbar_expect_tx_e(&sm.q_full, kTileBytes);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_4d_e(sm.q + bx * kHalfBytes, &tmQ, &sm.q_full, kBoxCols * bx, h_first, qs0, un.b);
      }
    }
    if (kAhead && ok)  // the last tile's V
      for (int part = 0; part < kParts && ok; ++part) ok = load_entry(&tmV, __ldg(list + n - 1) >> 1, part);
    // Never leave copies in flight.
    for (int u = max(0, t - kStages); u < t; ++u) {
      int dummy = 0;
      mbar_wait(&sm.kv_full[u % kStages], (u / kStages) & 1, &dummy, gstatus,
                LCATTN_ERR_DEVICE_TIMEOUT);
    }
    if (t > 0) {
      int dummy = 0;
      mbar_wait(&sm.q_full, 0, &dummy, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
    }
  } else if (warp == 5 && n > 0) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t idesc_qk = F8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
    const uint32_t idesc_pv = F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D / kParts, false, true);
    const uint64_t dq = sdesc_sw128(smem_u32(sm.q), 16, 1024);
    const uint64_t dk0 = sdesc_sw128(smem_u32(sm.kv[0]), 16, 1024);
    // V tile read MN-major (bf16), or V^T tile read K-major (e4m3).
    const uint64_t dv0 = sdesc_sw128(smem_u32(sm.kv[0]), F8 ? 16u : static_cast<uint32_t>(kHalfBytes), 1024);
    // O (+)= P V: A = P from TMEM (8 columns per k-step), B = V (MN-major, 16
    // key rows per k-step) or V^T (K-major, 32 keys per k-step).
    auto gemm_pv = [&](uint32_t tOp, uint32_t tP, uint64_t vb, uint32_t acc) {
      if constexpr (F8) {
        mma8_ts_er(tOp, tP, vb, idesc_pv, acc);
        #pragma unroll
        for (int kk = 1; kk < SplitGeom<D, F8>::kPvSteps; ++kk)
          mma8_ts_er(tOp, tP + kk * 8, sdesc_add(vb, kk * 32), idesc_pv, 1u);
      } else {
        mma_ts_er(tOp, tP, vb, idesc_pv, acc);
        #pragma unroll
        for (int kk = 1; kk < SplitGeom<D, F8>::kPvSteps; ++kk)
          mma_ts_e<1>(tOp, tP + kk * 8, sdesc_add(vb, kk * 2048), idesc_pv);
      }
    };
    // S (+)= Q K^T over one ring entry: k-steps of 32 bytes, the next box after four.
    auto gemm_s = [&](uint32_t tS, uint64_t qp, uint64_t kb, bool first) {
      if constexpr (F8) {
        if (first) mma8_ss_e<0>(tS, qp, kb, idesc_qk);
        else mma8_ss_e<1>(tS, qp, kb, idesc_qk);
      } else {
        if (first) mma_ss_e<0>(tS, qp, kb, idesc_qk);
        else mma_ss_e<1>(tS, qp, kb, idesc_qk);
      }
      #pragma unroll
      for (int kk = 1; kk < SplitGeom<D, F8>::kSSteps; ++kk) {
        const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
        if constexpr (F8) mma8_ss_e<1>(tS, sdesc_add(qp, off), sdesc_add(kb, off), idesc_qk);
        else mma_ss_e<1>(tS, sdesc_add(qp, off), sdesc_add(kb, off), idesc_qk);
      }
    };
    const uint32_t tO = tmem + 256;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full, 0, abort_flag, gstatus,
                                                LCATTN_ERR_DEVICE_TIMEOUT));
    // PV(tt): O (+)= P(tt) V(tt), once the softmax has released P(tt).
    auto issue_pv = [&](int tt) -> bool {
      bool okw = mbar_wait(&sm.p_full[tt & 1], (tt >> 1) & 1, abort_flag, gstatus,
                           LCATTN_ERR_DEVICE_TIMEOUT);
      const uint32_t tP = tmem + (tt & 1) * 128;
      #pragma unroll 1
      for (int part = 0; part < kParts; ++part) {  // V entries: columns [part * D/kParts, ...) of O
        const int tv = !kAhead || tt == n - 1 ? kE * tt + kParts + part : kE * tt + kE + part;
        if (okw) okw = mbar_wait(&sm.kv_full[tv % kStages], (tv / kStages) & 1, abort_flag, gstatus,
                                 LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, okw)) return false;
        tc_fence_after();
        const uint64_t vb = sdesc_add(dv0, (tv % kStages) * kEntryBytes);
        const uint32_t tOp = tO + part * (D / kParts);
        gemm_pv(tOp, tP, vb, tt > 0 ? 1u : 0u);
        tc_commit_e(&sm.kv_empty[tv % kStages]);
      }
      tc_commit_e(&sm.o_full);
      if (tt == n - 1) tc_commit_e(&sm.o_done);
      return true;
    };
    if (ok) tc_fence_after();
    for (int j = 0; ok && j < n; ++j) {
      const uint32_t tS = tmem + (j & 1) * 128;
      #pragma unroll 1
      for (int part = 0; part < kParts; ++part) {  // K entries: head-dim parts of the tile
        const int tk = !kAhead ? kE * j + part : (j == 0 ? part : kE * j - kParts + part);
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.kv_full[tk % kStages], (tk / kStages) & 1,
                                               abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT));
        if (!ok) break;
        tc_fence_after();
        const uint64_t kb = sdesc_add(dk0, (tk % kStages) * kEntryBytes);
        const uint64_t qp = sdesc_add(dq, part * kEntryBytes);
        gemm_s(tS, qp, kb, part == 0);
        tc_commit_e(&sm.kv_empty[tk % kStages]);
      }
      if (!ok) break;
      tc_commit_e(&sm.s_full[j & 1]);
      if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
    }
    if (ok) issue_pv(n - 1);
    tc_commit_e(&sm.drain);
    int dummy = 0;
    mbar_wait(&sm.drain, 0, &dummy, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    const int r = tid;  // TMEM lane = packed row
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t tO = tmem + lane_off + 256;
    const int s_pos = qs0 + r / a.Gp;            // query position of this row
    const int h = h_first + r % a.Gp;
    const float sl2 = a.scale_log2;
    const int last_kt = (pr.Sk - 1) / kBN;
    const bool ragged_k = (pr.Sk % kBN) != 0;
    const bool use_rows = a.mask.row_bounds != nullptr;
    int4 rb = make_int4(0, 0, 0, 0);
    if (use_rows && s_pos < pr.Sq) rb = __ldg(a.mask.row_bounds + (int64_t)un.b * pr.Sq + s_pos);
    float m_run = -INFINITY, l_run = 0.f;
    // A warp whose 32 packed rows all lie past the last query position (decode
    // rows fill 1/Rq of a tile) only keeps the barriers in step: it stages its
    // share of the column bounds and releases P without computing it.  Its O
    // rows are never written out.
    const bool warp_live = __any_sync(0xffffffffu, s_pos < pr.Sq);
    bool ok = true;
    int n_partial = 0;
    for (int j = 0; j < n; ++j) {
      const int e = __ldg(list + j);
      const int kt = e >> 1;
      const bool partial = (e & 1) != 0;
      const bool masked = partial || (ragged_k && kt == last_kt);
      uint32_t mw[4] = {0u, 0u, 0u, 0u};
      const int j0 = kt * kBN, j1 = min(pr.Sk, j0 + kBN);
      if (masked && partial && use_rows) {
        const int lo0 = max(rb.x, j0) - j0, hi0 = min(rb.y, j1) - j0;
        const int lo1 = max(rb.z, j0) - j0, hi1 = min(rb.w, j1) - j0;
        #pragma unroll
        for (int w = 0; w < 4; ++w) mw[w] = range_bits(lo0, hi0, 32 * w) | range_bits(lo1, hi1, 32 * w);
      } else if (masked && partial) {
        // The tile's 128 column bounds, staged once for all rows.
        const int u = n_partial & 1;
        const int key = j0 + r;
        sm.bnd[u][r] = key < pr.Sk ? __ldg(a.mask.col_bounds + (int64_t)un.b * pr.Sk + key)
                                   : make_int4(0, 0, 0, 0);
        mbar_arrive(&sm.bnd_ready[u]);
        ok = mbar_wait(&sm.bnd_ready[u], (n_partial >> 1) & 1, abort_flag, gstatus,
                       LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        ++n_partial;
        #pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t bits = 0u;
          #pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int4 v = sm.bnd[u][32 * w + c];
            const bool allow = (v.x <= s_pos && s_pos < v.y) || (v.z <= s_pos && s_pos < v.w);
            bits |= (allow ? 1u : 0u) << c;
          }
          mw[w] = bits;
        }
      } else if (masked) {  // a full tile cut by the end of the key sequence
        #pragma unroll
        for (int w = 0; w < 4; ++w) mw[w] = range_bits(0, j1 - j0, 32 * w);
      }
      const int sb = j & 1;
      const uint32_t tS = tmem + lane_off + sb * 128;
      ok = mbar_wait(&sm.s_full[sb], (j >> 1) & 1, abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      if (!warp_live) {  // (waiting for S(j) keeps this warp's arrivals on P(j)'s phase)
        mbar_arrive(&sm.p_full[sb]);
        continue;
      }
      tc_fence_after();
      uint32_t xr[128];
      tmem_ld32(tS + 0, xr + 0);
      tmem_ld32(tS + 32, xr + 32);
      tmem_ld32(tS + 64, xr + 64);
      tmem_ld32(tS + 96, xr + 96);
      tmem_ld_wait();
      float x[128];
      #pragma unroll
      for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(xr[c]);
      if (masked) {
        #pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!((mw[c >> 5] >> (c & 31)) & 1u)) x[c] = -INFINITY;
      }
      float m4[4];
      #pragma unroll
      for (int c = 0; c < 4; ++c) m4[c] = fmaxf(x[2 * c], x[2 * c + 1]);
      #pragma unroll
      for (int c = 8; c < 128; c += 2) m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], x[c], x[c + 1]);
      const float m_tile = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]) * sl2;
      const bool need = m_tile > m_run + SplitGeom<D, F8>::kRescaleThreshold;
      const bool warp_rescale = __any_sync(0xffffffffu, need) && j > 0;
      const float m_new = need ? m_tile : m_run;
      const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;
      m_run = m_new;
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // e4m3 P is P * 2^kLog2PScale, the shift folded into the exponent; l carries
      // the same factor, which cancels in O / l.
      const float negm_s = -(m_use - SplitGeom<D, F8>::kLog2PScale);
      const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(negm_s, negm_s);
      float2 s4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      if constexpr (F8) {
        uint32_t pk[32];  // four keys per column
        #pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 y0 = fma2(make_float2(x[4 * i], x[4 * i + 1]), sl2v, negm);
          const float2 y1 = fma2(make_float2(x[4 * i + 2], x[4 * i + 3]), sl2v, negm);
          const float2 p0 = make_float2(fast_exp2(y0.x), fast_exp2(y0.y));
          const float2 p1 = make_float2(fast_exp2(y1.x), fast_exp2(y1.y));
          s4[i & 3] = add2(s4[i & 3], add2(p0, p1));
          pk[i] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
        }
        tmem_st32(tS, pk);
      } else {
        #pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[32];
          #pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 y = fma2(make_float2(x[c * 64 + 2 * i], x[c * 64 + 2 * i + 1]), sl2v, negm);
            const float2 p = make_float2(fast_exp2(y.x), fast_exp2(y.y));
            s4[i & 3] = add2(s4[i & 3], p);
            pk[i] = pack_bf16x2(p.x, p.y);
          }
          tmem_st32(tS + c * 32, pk);
        }
      }
      const float2 s2 = add2(add2(s4[0], s4[1]), add2(s4[2], s4[3]));
      l_run = l_run * alpha + (s2.x + s2.y);
      if (warp_rescale) {
        // O holds PV up to tile j-1 once that PV completes; scale it in place
        // before P(j) is released (PV(j) waits for that release).
        ok = mbar_wait(&sm.o_full, (j - 1) & 1, abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        #pragma unroll (D <= 128 ? D / 32 : 1)
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o32[32];
          tmem_ld32(tO + c * 32, o32);
          tmem_ld_wait();
          #pragma unroll
          for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
          tmem_st32(tO + c * 32, o32);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[sb]);
    }
    // ---- epilogue: O / l (fp32) and the slice's LSE
    bool have_o = ok && n > 0;
    if (have_o) {
      have_o = __all_sync(0xffffffffu, mbar_wait(&sm.o_done, 0, abort_flag, gstatus,
                                                 LCATTN_ERR_DEVICE_TIMEOUT));
      tc_fence_after();
    }
    if (ok && warp_live && (have_o || n == 0)) {
      const bool live = l_run > 0.f;
      const float inv = live ? a.o_scale / l_run : 0.f;
      // O in batches that fit the registers (all of it up to D = 128).
      constexpr int kBatch = D <= 128 ? D : 32;
      float4* dst = reinterpret_cast<float4*>(
          a.o_part + ((((int64_t)un.c * pr.B + un.b) * pr.Sq + s_pos) * pr.Hq + h) * D);
      #pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += kBatch) {
        uint32_t o32[kBatch];
        if (have_o) {
          #pragma unroll
          for (int c = 0; c < kBatch / 32; ++c) tmem_ld32(tO + c0 + c * 32, o32 + c * 32);
          tmem_ld_wait();
        } else {
          #pragma unroll
          for (int i = 0; i < kBatch; ++i) o32[i] = 0u;
        }
        if (s_pos < pr.Sq) {
          #pragma unroll
          for (int i = 0; i < kBatch / 4; ++i)
            dst[c0 / 4 + i] = make_float4(__uint_as_float(o32[4 * i]) * inv, __uint_as_float(o32[4 * i + 1]) * inv,
                                          __uint_as_float(o32[4 * i + 2]) * inv, __uint_as_float(o32[4 * i + 3]) * inv);
        }
      }
      if (s_pos < pr.Sq) {
        a.lse_part[(((int64_t)un.c * pr.B + un.b) * pr.Hq + h) * pr.Sq + s_pos] =
            live ? (m_run - SplitGeom<D, F8>::kLog2PScale + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per (batch, query position, head): merge the slices.  Lane l owns
// columns [l * D/32, (l + 1) * D/32).
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(SplitArgs a) {
  constexpr int kPer = D / 32;
  const ProblemDev& pr = a.pr;
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)pr.B * pr.Sq * pr.Hq;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t per_split_o = (int64_t)pr.B * pr.Sq * pr.Hq * D;
  const int64_t per_split_l = (int64_t)pr.B * pr.Hq * pr.Sq;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += stride) {
    const int h = (int)(w % pr.Hq);
    const int s = (int)((w / pr.Hq) % pr.Sq);
    const int b = (int)(w / ((int64_t)pr.Hq * pr.Sq));
    const int64_t li = ((int64_t)b * pr.Hq + h) * pr.Sq + s;
    float m = -INFINITY;
    for (int c = 0; c < a.splits; ++c) m = fmaxf(m, a.lse_part[c * per_split_l + li]);
    float acc[kPer];
    #pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int c = 0; c < a.splits; ++c) {
        const float l = a.lse_part[c * per_split_l + li];
        if (l == -INFINITY) continue;
        const float wgt = __expf(l - m);
        const float* o = a.o_part + c * per_split_o + w * D + lane * kPer;
        #pragma unroll
        for (int i = 0; i < kPer; ++i) acc[i] += wgt * o[i];
        wsum += wgt;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.o_sb +
                          (int64_t)s * a.o_ss + (int64_t)h * a.o_sh + lane * kPer;
    #pragma unroll
    for (int i = 0; i < kPer; i += 2)
      reinterpret_cast<uint32_t*>(orow)[i / 2] = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    if (lane == 0) a.lse[li] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
  }
}

}  // namespace

int split_heads_packed(int G) {
  int gp = 1;
  while (gp * 2 <= 128 && G % (gp * 2) == 0) gp *= 2;
  return gp;
}

namespace {

template <int D, bool F8 = false>
cudaError_t launch_split_d(const CUtensorMap& tq_packed, const CUtensorMap& tk,
                           const CUtensorMap& tv, const SplitArgs& a, cudaStream_t st) {
  static bool attr_done = false;
  const size_t smem = sizeof(SplitSmem<D, F8>) + 1024;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(split_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t units = (int64_t)a.pr.B * a.pr.Hkv * (a.pr.G / a.Gp) * a.nQc * a.splits;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  split_kernel<D, F8><<<(unsigned)units, kThreads, smem, st>>>(tq_packed, tk, tv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 152 * 32) blocks = 152 * 32;
  combine_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_split(const CUtensorMap& tq_packed, const CUtensorMap& tk,
                             const CUtensorMap& tv, const SplitArgs& a, cudaStream_t st) {
  if (a.pr.D == 64) return launch_split_d<64>(tq_packed, tk, tv, a, st);
  if (a.pr.D == 256) return launch_split_d<256>(tq_packed, tk, tv, a, st);
  return launch_split_d<128>(tq_packed, tk, tv, a, st);
}

cudaError_t launch_fwd_split_e4m3(const CUtensorMap& tq_packed, const CUtensorMap& tk, const CUtensorMap& tvt,
                                  const SplitArgs& a, cudaStream_t st) {
  if (a.pr.D != 128) return cudaErrorInvalidValue;
  return launch_split_d<128, true>(tq_packed, tk, tvt, a, st);
}

}  // namespace lcattn
