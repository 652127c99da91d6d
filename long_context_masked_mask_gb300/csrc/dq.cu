// dQ of masked attention for sm_103a, one CTA per (query tile, query head,
// batch): the query side of the backward computed on its own, so that no fp32
// reductions into a global accumulator are needed.  For every non-empty key
// tile j of the query tile's list it recomputes
//   S = Q K_j^T,  P' = scale * exp(S - LSE)  (masked entries 0),
//   dP = dO V_j^T,  dS' = P' (dP - D)   (D = rowsum(dO * O) from the pre-pass),
// and accumulates dQ += dS' K_j in tensor memory; the bf16 dQ tile is written
// once at the end.  The key side (dK, dV) comes from the dK/dV kernel built
// without its dQ product.  The gradients are the textbook ones for L = <O, dO>
// of the attention operator the pages benchmark ("Long-Context Attention
// Benchmark", xllm-io blog review, sections "密集注意力内核" and "稀疏注意力内核";
// sections "稀疏内核性能" and "核心发现总结" single the backward out as the main
// bottleneck).
//
// Roles (384 threads, 3 warpgroups):
//   warps 0-3, 4-7  elementwise, one warpgroup per half (64 keys) of a tile's
//              128 key columns; thread r is query row r (TMEM lane r).  It
//              forms P' from S, then dS' from dP, and writes dS' (bf16) over
//              its S columns, where the dQ product reads it as the A operand.
//              At the end they store dQ (warpgroup x: head-dim half x).
//   warp  8    producer: Q and dO once, K_j through a 3-stage ring and V_j
//              through a 2-stage ring (V is released after dP, K after dQ).
//   warp  9    TMEM owner and MMA issuer; warps 10-11 idle (they complete the
//              warpgroup for setmaxnreg).
// TMEM: [0,128) S / dS' buffer 0 | [128,256) buffer 1 | [256,384) dP |
//       [384, 384+D) dQ.
// MMA order per key tile j (S(0), dP(0), S(1) first):
//   wait dP(j) read -> dP(j+1) | wait dS'(j) -> dQ += dS'(j) K_j -> release K_j |
//   S(j+2) into the buffer dS'(j) used (the dQ product reads it first, in order).
#include <cuda_bf16.h>

#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

using namespace dev;

constexpr int kThreadsDq = 384;
constexpr int kHalf = 16384;     // one 64-column box of a 128-row bf16 tile
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kRegsDqWork = 216;
constexpr int kRegsDqCtl = 72;
static_assert(128 * (2 * kRegsDqWork + kRegsDqCtl) <= kThreadsDq * 168, "register split");
constexpr float kLog2eDq = 1.4426950408889634f;

template <int D>
struct DqSmem {
  static constexpr int kTile = 128 * D * 2;
  alignas(1024) uint8_t q[kTile];
  alignas(1024) uint8_t dO[kTile];
  alignas(1024) uint8_t k[kKStages][kTile];
  alignas(1024) uint8_t v[kVStages][kTile];
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], dp_full, dp_free, ds_ready, done;
  uint32_t tmem_base;
  int abort_flag;
};

struct DqKernelArgs {
  BwdArgs a;
};

__device__ __forceinline__ int dq_block_of(const int32_t* offs, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bits [lo, hi) of a 64-bit key mask that fall into the word starting at `base`.
__device__ __forceinline__ uint32_t dq_range_bits(int lo, int hi, int base) {
  const int a = max(lo, base), b = min(hi, base + 32);
  if (b <= a) return 0u;
  const int n = b - a;
  return (n == 32) ? 0xffffffffu : (((1u << n) - 1u) << (a - base));
}

// Allowed-key bits of query row `row` for keys [k0, k0 + 64) (bit c = key k0 + c),
// keys past Sk excluded.  `rb` holds the row's key intervals when the
// descriptor carries row bounds; `qb_row` is the row's query block for block maps.
__device__ __forceinline__ void dq_row_mask(const MaskDev& m, const ProblemDev& pr, int b, int h, int row,
                                            int qb_row, bool use_rows, int4 rb, int k0,
                                            uint32_t& m0, uint32_t& m1) {
  const int k1 = min(k0 + 64, pr.Sk);
  m0 = m1 = 0u;
  if (k1 <= k0 || row >= pr.Sq) return;
  if (m.kind == LCATTN_MASK_COLBOUNDS) {
    if (use_rows) {
      const int lo0 = max(rb.x, k0) - k0, hi0 = min(min(rb.y, k1), k0 + 64) - k0;
      const int lo1 = max(rb.z, k0) - k0, hi1 = min(min(rb.w, k1), k0 + 64) - k0;
      m0 = dq_range_bits(lo0, hi0, 0) | dq_range_bits(lo1, hi1, 0);
      m1 = dq_range_bits(lo0, hi0, 32) | dq_range_bits(lo1, hi1, 32);
    } else {
      // Column bounds only: test this row against each key's two intervals.
      const int4* cb = m.col_bounds + (int64_t)b * pr.Sk;
      for (int c = 0; c < k1 - k0; ++c) {
        const int4 v = __ldg(cb + k0 + c);
        const bool ok = (v.x <= row && row < v.y) || (v.z <= row && row < v.w);
        if (ok) {
          if (c < 32) m0 |= 1u << c; else m1 |= 1u << (c - 32);
        }
      }
    }
  } else {
    const uint8_t* map = m.block_map + (((int64_t)b * pr.Hq + h) * m.nQb + qb_row) * (int64_t)m.nKb;
    for (int kb = dq_block_of(m.k_offs, m.nKb, k0); kb < m.nKb; ++kb) {
      const int lo = max(__ldg(m.k_offs + kb), k0);
      if (lo >= k1) break;
      const int hi = min(__ldg(m.k_offs + kb + 1), k1);
      if (hi > lo && __ldg(map + kb)) {
        m0 |= dq_range_bits(lo - k0, hi - k0, 0);
        m1 |= dq_range_bits(lo - k0, hi - k0, 32);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsDq, 1)
dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
          const __grid_constant__ DqKernelArgs ka) {
  constexpr int kTile = DqSmem<D>::kTile;
  constexpr int kBoxes = D / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const BwdArgs& a = ka.a;
  const ProblemDev& pr = a.pr;
  int32_t* gstatus = a.meta.status;
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(gstatus, 0, LCATTN_ERR_CUDA);
    return;
  }
  DqSmem<D>& sm = *reinterpret_cast<DqSmem<D>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Unit: (order index, head within the KV group) in blockIdx.x, so the query
  // heads of one group that share a key list run side by side; KV head in y,
  // batch in z.  Longest lists first (the mask compiler's forward order).
  const int b = blockIdx.z;
  const int g = blockIdx.y;
  const int hl = (int)(blockIdx.x % pr.G);
  const int oi = (int)(blockIdx.x / pr.G);
  const int h = g * pr.G + hl;
  const int lh = a.meta.nH == 1 ? 0 : h;
  const int64_t bh = (int64_t)b * a.meta.nH + lh;
  const int qt = __ldg(a.meta.fwd_ord + bh * a.meta.nQt + oi);
  const int n = __ldg(a.meta.fwd_cnt + bh * a.meta.nQt + qt);
  const int32_t* lst = a.meta.fwd_lst + (bh * a.meta.nQt + qt) * a.meta.nKt;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kKStages; ++s) { mbar_init(&sm.k_full[s], 1); mbar_init(&sm.k_empty[s], 1); }
    for (int s = 0; s < kVStages; ++s) { mbar_init(&sm.v_full[s], 1); mbar_init(&sm.v_empty[s], 1); }
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_full[1], 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.dp_free, 256);
    mbar_init(&sm.ds_ready, 256);
    mbar_init(&sm.done, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  const int TO = LCATTN_ERR_DEVICE_TIMEOUT;

  if (warp >= 8) {
    regs_dec<kRegsDqCtl>();
    if (warp == 8 && n > 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
      }
      __syncwarp();
      mbar_expect_tx_e(&sm.q_full, 2 * kTile);
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_load_4d_e(sm.q + bx * kHalf, &tmQ, &sm.q_full, 64 * bx, h, qt * kBM, b);
        tma_load_4d_e(sm.dO + bx * kHalf, &tmdO, &sm.q_full, 64 * bx, h, qt * kBM, b);
      }
      // K runs up to two tiles ahead of V (S(j+2) is issued before dP(j+2)):
      // load K(j), then V(j), with each ring's own empty barriers.
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n; ++j) {
        const int kt = __ldg(lst + j) >> 1;
        const int sk = j % kKStages, sv = j % kVStages;
        if (j >= kKStages) {
          const bool ok = mbar_wait(&sm.k_empty[sk], ((j / kKStages) - 1) & 1, abort_flag, gstatus, TO);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        mbar_expect_tx_e(&sm.k_full[sk], kTile);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_4d_e(sm.k[sk] + bx * kHalf, &tmK, &sm.k_full[sk], 64 * bx, g, kt * kBN, b);
        issued_k = j + 1;
        if (j >= kVStages) {
          const bool ok = mbar_wait(&sm.v_empty[sv], ((j / kVStages) - 1) & 1, abort_flag, gstatus, TO);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        mbar_expect_tx_e(&sm.v_full[sv], kTile);
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_load_4d_e(sm.v[sv] + bx * kHalf, &tmV, &sm.v_full[sv], 64 * bx, g, kt * kBN, b);
        issued_v = j + 1;
      }
      // Let every copy in flight land before the CTA may exit.
      int dummy = 0;
      mbar_wait(&sm.q_full, 0, &dummy, gstatus, TO);
      for (int t = max(0, issued_k - kKStages); t < issued_k; ++t)
        mbar_wait(&sm.k_full[t % kKStages], (t / kKStages) & 1, &dummy, gstatus, TO);
      for (int t = max(0, issued_v - kVStages); t < issued_v; ++t)
        mbar_wait(&sm.v_full[t % kVStages], (t / kVStages) & 1, &dummy, gstatus, TO);
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t id_kmaj = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_ts = idesc_bf16_f32(128, D, false, true);
      const uint32_t tdP = tmem + 256, tdQ = tmem + 384;
      const uint64_t dQ_k = sdesc_sw128(smem_u32(sm.q), 16, 1024);
      const uint64_t dO_k = sdesc_sw128(smem_u32(sm.dO), 16, 1024);
      const uint64_t dK_k = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(smem_u32(sm.k[0]), kHalf, 1024);
      const uint64_t dV_k = sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
      // Both operands K-major (contraction over the head dim).
      auto issue_kmaj = [&](uint32_t d, uint64_t a0, uint64_t b0) {
        mma_ss_e<0>(d, a0, b0, id_kmaj);
        #pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_ss_e<1>(d, sdesc_add(a0, off), sdesc_add(b0, off), id_kmaj);
        }
      };
      bool ok = true;
      if (n > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full, 0, abort_flag, gstatus, TO)) &&
             __all_sync(0xffffffffu, mbar_wait(&sm.k_full[0], 0, abort_flag, gstatus, TO));
        if (ok) {
          tc_fence_after();
          issue_kmaj(tmem, dQ_k, dK_k);  // S(0)
          tc_commit_e(&sm.s_full[0]);
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[0], 0, abort_flag, gstatus, TO));
        }
        if (ok) {
          tc_fence_after();
          issue_kmaj(tdP, dO_k, dV_k);   // dP(0)
          tc_commit_e(&sm.dp_full);
          tc_commit_e(&sm.v_empty[0]);
          if (n > 1) {
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[1], 0, abort_flag, gstatus, TO));
            if (ok) {
              tc_fence_after();
              issue_kmaj(tmem + 128, dQ_k, sdesc_add(dK_k, kTile));  // S(1)
              tc_commit_e(&sm.s_full[1]);
            }
          }
        }
      }
      for (int j = 0; ok && j < n; ++j) {
        // dP(j+1) once the elementwise warps hold dP(j) in registers.
        if (j + 1 < n) {
          const int sv = (j + 1) % kVStages;
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.dp_free, j & 1, abort_flag, gstatus, TO)) &&
               __all_sync(0xffffffffu, mbar_wait(&sm.v_full[sv], ((j + 1) / kVStages) & 1, abort_flag,
                                                 gstatus, TO));
          if (!ok) break;
          tc_fence_after();
          issue_kmaj(tdP, dO_k, sdesc_add(dV_k, sv * kTile));
          tc_commit_e(&sm.dp_full);
          tc_commit_e(&sm.v_empty[sv]);
        }
        // dQ += dS'(j) K_j: A = dS' from TMEM (keys 0-63 in the first 32
        // columns of each half's region, 64-127 at +64), B = K_j MN-major.
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.ds_ready, j & 1, abort_flag, gstatus, TO));
        if (!ok) break;
        tc_fence_after();
        {
          const int sk = j % kKStages;
          const uint32_t tS = tmem + (j & 1) * 128;
          const uint64_t bk = sdesc_add(dK_mn, sk * kTile);
          mma_ts_er(tdQ, tS, bk, id_ts, j > 0 ? 1u : 0u);
          #pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ts_e<1>(tdQ, tS + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_add(bk, kk * 2048), id_ts);
          tc_commit_e(&sm.k_empty[sk]);
        }
        // S(j+2) into the buffer dS'(j) occupied (read by the dQ product above, in order).
        if (j + 2 < n) {
          const int sk2 = (j + 2) % kKStages;
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[sk2], ((j + 2) / kKStages) & 1, abort_flag,
                                                 gstatus, TO));
          if (!ok) break;
          tc_fence_after();
          issue_kmaj(tmem + (j & 1) * 128, dQ_k, sdesc_add(dK_k, sk2 * kTile));
          tc_commit_e(&sm.s_full[j & 1]);
        }
      }
      tc_commit_e(&sm.done);
      int dummy = 0;
      mbar_wait(&sm.done, 0, &dummy, gstatus, TO);
    }
  } else {
    regs_inc<kRegsDqWork>();
    // ------------------------------------------------------------ elementwise
    const int x = warp >> 2;                  // key half of the tile
    const int r = 32 * (warp & 3) + lane;     // query row within the tile (TMEM lane)
    const int c0 = 64 * x;
    const int row = qt * kBM + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float sl2 = a.scale_log2;
    // Per-row constants: the exponent addend -(LSE log2 e - log2 scale) (-inf where
    // P' must be 0: rows past Sq and rows that allow nothing) and -D.
    float l2 = -INFINITY, nd = 0.f;
    if (row < pr.Sq) {
      const float l = __ldg(a.lse + ((int64_t)b * pr.Hq + h) * pr.Sq + row);
      l2 = (l == -INFINITY) ? -INFINITY : log2f(a.scale) - l * kLog2eDq;
      nd = -__ldg(a.dvec + ((int64_t)b * pr.Hq + h) * pr.Sq + row);
    }
    const bool use_rows = a.mask.kind == LCATTN_MASK_COLBOUNDS && a.mask.row_bounds != nullptr;
    int4 rb = make_int4(0, 0, 0, 0);
    int qb_row = 0;
    if (row < pr.Sq) {
      if (use_rows) rb = __ldg(a.mask.row_bounds + (int64_t)b * pr.Sq + row);
      if (a.mask.kind == LCATTN_MASK_BLOCKMAP) qb_row = dq_block_of(a.mask.q_offs, a.mask.nQb, row);
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int e = __ldg(lst + j);
      const int kt = e >> 1;
      const int k0 = kt * kBN + c0;
      const bool masked = (e & 1) != 0 || kt * kBN + kBN > pr.Sk;
      uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
      if (masked) dq_row_mask(a.mask, pr, b, h, row, qb_row, use_rows, rb, k0, m0, m1);
      const uint32_t tS = tmem + lane_off + (j & 1) * 128;
      ok = mbar_wait(&sm.s_full[j & 1], (j >> 1) & 1, abort_flag, gstatus, TO);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // ---- P' = scale * P for 64 keys, kept packed in registers
      uint32_t pk[32];
      {
        uint32_t s0[32], s1[32];
        tmem_ld32(tS + c0, s0);
        tmem_ld32(tS + c0 + 32, s1);
        tmem_ld_wait();
        const float2 sl2v = make_float2(sl2, sl2), l2v = make_float2(l2, l2);
        #pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          const float2 ya = fma2(make_float2(__uint_as_float(s0[2 * c2]), __uint_as_float(s0[2 * c2 + 1])), sl2v, l2v);
          const float2 yb = fma2(make_float2(__uint_as_float(s1[2 * c2]), __uint_as_float(s1[2 * c2 + 1])), sl2v, l2v);
          float pa0 = fast_exp2(ya.x), pa1 = fast_exp2(ya.y), pb0 = fast_exp2(yb.x), pb1 = fast_exp2(yb.y);
          if (masked) {
            pa0 = ((m0 >> (2 * c2)) & 1u) ? pa0 : 0.f;
            pa1 = ((m0 >> (2 * c2 + 1)) & 1u) ? pa1 : 0.f;
            pb0 = ((m1 >> (2 * c2)) & 1u) ? pb0 : 0.f;
            pb1 = ((m1 >> (2 * c2 + 1)) & 1u) ? pb1 : 0.f;
          }
          pk[c2] = pack_bf16x2(pa0, pa1);
          pk[16 + c2] = pack_bf16x2(pb0, pb1);
        }
      }
      // ---- dS' = P' (dP - D), from the bf16 P'
      ok = mbar_wait(&sm.dp_full, j & 1, abort_flag, gstatus, TO);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t dsk[32];
      {
        uint32_t d0[32], d1[32];
        tmem_ld32(tmem + lane_off + 256 + c0, d0);
        tmem_ld32(tmem + lane_off + 256 + c0 + 32, d1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&sm.dp_free);  // dP(j+1) may overwrite the dP columns now
        const float2 ndv = make_float2(nd, nd);
        // dP - D on column pairs (fp32), rounded to bf16 pairs, times the bf16 P'
        // pairs on the packed bf16 ALU (dS' leaves in bf16 either way).
        #pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          const float2 ta = add2(make_float2(__uint_as_float(d0[2 * c2]), __uint_as_float(d0[2 * c2 + 1])), ndv);
          const float2 tb = add2(make_float2(__uint_as_float(d1[2 * c2]), __uint_as_float(d1[2 * c2 + 1])), ndv);
          dsk[c2] = mul_bf16x2(pk[c2], pack_bf16x2(ta.x, ta.y));
          dsk[16 + c2] = mul_bf16x2(pk[16 + c2], pack_bf16x2(tb.x, tb.y));
        }
      }
      tmem_st32(tS + c0, dsk);  // columns [64x, 64x + 32) of this S buffer: only this warpgroup's
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.ds_ready);
    }
    // ---- dQ out (warpgroup x: head dims [x D/2, (x+1) D/2)), bf16; zero for an empty list.
    // The TMEM loads are warp-collective: every lane runs them, and only the
    // stores are limited to rows inside the sequence.
    if (ok) {
      bool have = n > 0;
      if (have) {
        have = __all_sync(0xffffffffu, mbar_wait(&sm.done, 0, abort_flag, gstatus, TO));
        tc_fence_after();
      }
      if (have || n == 0) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.dq) + (int64_t)b * a.q_sb +
                             (int64_t)row * a.q_ss + (int64_t)h * a.q_sh + x * (D / 2);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t xr[32];
          if (n > 0) {
            tmem_ld32(tmem + lane_off + 384 + x * (D / 2) + c * 32, xr);
            tmem_ld_wait();
          } else {
            #pragma unroll
            for (int k = 0; k < 32; ++k) xr[k] = 0u;
          }
          if (row < pr.Sq) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
            #pragma unroll
            for (int u = 0; u < 4; ++u)
              d4[u] = make_uint4(pack_bf16x2(__uint_as_float(xr[8 * u]), __uint_as_float(xr[8 * u + 1])),
                                 pack_bf16x2(__uint_as_float(xr[8 * u + 2]), __uint_as_float(xr[8 * u + 3])),
                                 pack_bf16x2(__uint_as_float(xr[8 * u + 4]), __uint_as_float(xr[8 * u + 5])),
                                 pack_bf16x2(__uint_as_float(xr[8 * u + 6]), __uint_as_float(xr[8 * u + 7])));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_dq_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
  static bool attr_done = false;
  const size_t smem = sizeof(DqSmem<D>);
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  DqKernelArgs ka;
  ka.a = a;
  dim3 grid(a.meta.nQt * a.pr.G, a.pr.Hkv, a.pr.B);
  dq_kernel<D><<<grid, kThreadsDq, smem, st>>>(tq, tk, tv, tdo, ka);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
  return a.pr.D == 64 ? launch_dq_d<64>(tq, tk, tv, tdo, a, st) : launch_dq_d<128>(tq, tk, tv, tdo, a, st);
}

}  // namespace lcattn
