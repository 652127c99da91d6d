// Forward masked attention for sm_103a.
//
// Computes O = softmax(scale * Q K^T restricted to the allowed keys) V and the
// natural-log LSE per query row -- the forward operator benchmarked on the
// pages ("Long-Context Attention Benchmark", xllm-io blog review, sections
// "密集注意力内核" and "密集内核性能": bf16, head dim 128, GQA 64:8 and MHA 64:64).
//
// Persistent: one CTA per SM walks a sequence of work items.  An item is up to
// two 128-row query tiles ("slots") that share one list of key tiles: two query
// heads of the same GQA group (the mask is head independent for column
// bounds), or a single tile otherwise.  With single-tile items (D <= 128) the
// items alternate between the two slots, so one slot's epilogue overlaps the
// other slot's first tiles.  Roles:
//   warps 0-3  softmax for slot 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax for slot 1
//   warp  8    TMA producer: per item its Q tiles, then K_j, V_j into a 4-deep
//              ring that runs on across items
//   warp  9    TMEM owner and single-thread tcgen05.mma issuer
//   warps 10-11 idle (they complete the third warpgroup for setmaxnreg)
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  The softmax
// writes P (bf16 pairs) over the first 64 columns of its S, and the PV product
// reads P from TMEM (A operand) and V from shared memory (B operand).
// Issue order per key tile j: PV0(j-1), S0(j), PV1(j-1), S1(j), so each slot's
// softmax overlaps the other slot's two GEMMs; the order runs on across items,
// so an item's tail (last PV, epilogue) overlaps the next item's first GEMMs.
// The running max is kept in the log2 domain and only moved when a row max grows
// by more than 8 (a factor 256 of headroom in fp32 / bf16), so O is rescaled in
// TMEM rarely; the final O is divided by the row sum in the epilogue.
#include <cuda_bf16.h>

#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

using namespace dev;

// Head dim D (64, 128 or 256) is a template parameter: a Q, K or V tile is 128
// rows x D bf16, loaded as D/64 boxes of 64 columns.  The K/V ring holds 128 KB.
// An entry is a whole K or V tile for D <= 128 (8 stages of 64-wide tiles, 4
// of 128-wide); at D = 256 a tile is two entries, its head-dim halves (4
// stages of 32 KB), so that the next tile's K streams in while this tile's
// halves are consumed.  At D = 256 an item is always one head (TMEM: two S
// buffers + a 256-column O) and there is one Q buffer.
// F8 (e4m3 inputs, D = 128 only): a tile is 128 rows x 128 bytes, one box, and
// the ring has 8 stages of 16 KB; the V entries are tiles of V^T (a 128 x 128
// block of the key-contiguous V^T written by a pre-pass), so that both
// kind::f8f6f4 operands of the PV product are K-major.
template <int D, bool F8 = false> struct FwdGeom {
  static_assert(!F8 || D == 128, "the e4m3 forward is built for head dim 128");
  static constexpr int kElem = F8 ? 1 : 2;                      // bytes per element
  static constexpr int kTileBytes = 128 * D * kElem;
  static constexpr int kBoxCols = F8 ? 128 : 64;                // elements per 128-byte box row
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kParts = D == 256 ? 2 : 1;            // ring entries per K (or V) tile
  static constexpr int kEntryBytes = kTileBytes / kParts;
  static constexpr int kBoxesPerEntry = kBoxes / kParts;
  static constexpr int kStages = (D == 64 || F8) ? 8 : 4;    // K/V ring depth (entries)
  static constexpr int kQBufs = D == 256 ? 1 : 2;
  // k-steps of the S product per entry (32 bytes of the contraction each) and
  // of the PV product per tile (16 keys for bf16 P, 32 for e4m3 P: 8 TMEM columns each).
  static constexpr int kSSteps = D * kElem / 32 / kParts;
  static constexpr int kPvSteps = F8 ? 4 : 8;
  // Largest P in the log2-domain online softmax: the running max moves only
  // when a row max grows by more than kRescaleThreshold, so P <= 2^threshold.
  // e4m3 P is stored as P * kPScale (at most 2^(4 + 4) = 256, inside e4m3's 448).
  static constexpr float kRescaleThreshold = F8 ? 4.0f : 8.0f;
  static constexpr float kPScale = F8 ? 16.0f : 1.0f;
};
constexpr int kItemQ = 4;           // depth of the work-item queue (producer -> other roles)
constexpr int kHalfBytes = 16384;   // one 64-column TMA box of 128 rows
constexpr int kThreads = 384;        // 3 warpgroups
// Register split (launch: 384 threads x 168): softmax warpgroups 200 each,
// producer/MMA warpgroup 104.  Same-box A/B against 216 / 72: one-head items
// 3-4% faster, head dim 64 1.3%, e4m3 0.5-1%, and, with the MMA warp's slot
// loop unrolled (which spilled at 72), bf16 two-head items 2.5-3.3%.
template <int D, int HPC, bool F8> struct FwdRegs {
  static constexpr int kSoftmax = 200;
  static constexpr int kOther = 104;
  static_assert(128 * (2 * kSoftmax + kOther) <= kThreads * 168, "register split");
};

template <int D, bool F8 = false>
struct FwdSmem {
  static constexpr int kStages = FwdGeom<D, F8>::kStages;
  static constexpr int kTileBytes = FwdGeom<D, F8>::kTileBytes;
  alignas(1024) uint8_t q[FwdGeom<D, F8>::kQBufs][kTileBytes];
  alignas(1024) uint8_t kv[kStages][FwdGeom<D, F8>::kEntryBytes];
  // Per slot: O staging for the epilogue's TMA stores (one 64-column box of
  // 128 rows, 128-byte swizzled).  Between epilogues its first 4 KB hold the
  // column bounds of partial tiles (two buffers of 128 int4).
  alignas(1024) uint8_t stg[2][kHalfBytes];
  uint64_t bnd_ready[2][2];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[4];  // per slot (two heads), per S buffer (one head), per slot and buffer (alternating)
  uint64_t p_full[2];
  uint64_t o_full[2];  // every PV into the slot's O has completed (one phase per PV)
  uint64_t o_last[2];  // an item's last PV into the slot's O has completed (one phase per item)
  uint64_t drain;
  uint64_t stg_full[2];  // a slot's staging box is written (128 arrivals; one phase per epilogue)
  uint64_t stg_free[2];  // ... and read by its TMA stores (one phase per epilogue)
  // Items handed from the producer to the other roles: (index, query tile, key
  // tiles, -); the producer has read the tile metadata, so the others need no
  // dependent global loads at an item's start.  Index -1 ends the sequence.
  int4 items[kItemQ];
  uint64_t item_full[kItemQ];
  uint64_t item_empty[kItemQ];
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdKernelArgs {
  FwdArgs a;
  int heads_per_cta;
  int head_block;  // one head per item: heads per block of the item order
  int total_items;
};

// Bits [lo, hi) of a 128-bit row mask that fall into the 32-bit word starting at `base`.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int base) {
  const int a = max(lo, base), b = min(hi, base + 32);
  if (b <= a) return 0u;
  const int n = b - a;
  return (n == 32) ? 0xffffffffu : (((1u << n) - 1u) << (a - base));
}

__device__ __forceinline__ int block_of(const int32_t* offs, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Allowed-key bits of query row `row` for key tile kt (bit c = key kt*128+c).
// Column bounds are read from `bnd` (the tile's 128 bounds in shared memory).
__device__ __forceinline__ void tile_mask_bits(const MaskDev& m, const ProblemDev& pr, int b,
                                               int h, int row, int qb_row, int kt,
                                               bool evaluate_mask, const int4* bnd,
                                               uint32_t (&mw)[4]) {
  const int j0 = kt * kBN;
  const int nvalid = min(kBN, pr.Sk - j0);
  mw[0] = mw[1] = mw[2] = mw[3] = 0u;
  if (!evaluate_mask) {  // full tile cut by the end of the key sequence
    mw[0] = range_bits(0, nvalid, 0);
    mw[1] = range_bits(0, nvalid, 32);
    mw[2] = range_bits(0, nvalid, 64);
    mw[3] = range_bits(0, nvalid, 96);
    return;
  }
  if (m.kind == LCATTN_MASK_COLBOUNDS) {
    // Bounds come from shared memory (staged by the caller); keys past the end
    // of the sequence were staged as empty intervals.
    #pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t bits = 0u;
      #pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int4 v = bnd[32 * w + c];
        const bool ok = (v.x <= row && row < v.y) || (v.z <= row && row < v.w);
        bits |= (ok ? 1u : 0u) << c;
      }
      mw[w] = bits;
    }
  } else {
    const int j1 = j0 + nvalid;
    const uint8_t* map =
        m.block_map + (((int64_t)b * pr.Hq + h) * m.nQb + qb_row) * (int64_t)m.nKb;
    uint32_t b0 = 0u, b1 = 0u, b2 = 0u, b3 = 0u;
    for (int kb = block_of(m.k_offs, m.nKb, j0); kb < m.nKb; ++kb) {
      const int lo = max(__ldg(m.k_offs + kb), j0);
      if (lo >= j1) break;
      const int hi = min(__ldg(m.k_offs + kb + 1), j1);
      if (hi > lo && __ldg(map + kb)) {
        b0 |= range_bits(lo - j0, hi - j0, 0);
        b1 |= range_bits(lo - j0, hi - j0, 32);
        b2 |= range_bits(lo - j0, hi - j0, 64);
        b3 |= range_bits(lo - j0, hi - j0, 96);
      }
    }
    mw[0] = b0; mw[1] = b1; mw[2] = b2; mw[3] = b3;
  }
}

// ---- persistent schedule ----------------------------------------------------
// An item is one query tile for `heads_per_cta` query heads.  Items are ordered
// rank-major: rank r is the r-th longest key-tile list of its (batch, head)
// list (the mask compiler's LPT order), so item costs fall along the sequence.
// CTAs take items greedily from a device-wide counter (longest-processing-time
// first): the producer warp fetches an index one item ahead (so it can warm L2
// with that item's query rows) and hands the indices to the MMA and softmax
// warps through a small queue in shared memory; -1 ends the sequence.

struct FwdItem {
  int b, h0, qt, n;
  const int32_t* list;
};

// idx < total_items < 2^31 (the launcher checks), so 32-bit arithmetic suffices.
// Two heads per item: rank-major over every (batch, head pair), so the items
// in flight share K/V through their KV group.  One head per item: items come
// in blocks of `hb` heads (whole GQA groups) of one batch entry, rank-major
// within a block; the items in flight then cover a few heads' K/V, which stays
// in L2 (with MHA every head has its own K/V, far more than L2 holds).
__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int hpc, int hb, int idx, int* rank_out = nullptr) {
  FwdItem it;
  int rank;
  if (hpc == 1) {
    const int per_block = hb * a.meta.nQt;
    const int blk = idx / per_block;
    const int r = idx - blk * per_block;
    rank = r / hb;
    const int nb = a.pr.Hq / hb;  // blocks per batch entry
    it.b = blk / nb;
    it.h0 = (blk - it.b * nb) * hb + (r - rank * hb);
  } else {
    const int groups = a.pr.Hq / hpc;
    const int per_rank = groups * a.pr.B;
    rank = idx / per_rank;
    const int rem = idx - rank * per_rank;
    it.b = rem / groups;
    it.h0 = (rem - it.b * groups) * hpc;
  }
  const int lh = a.meta.nH == 1 ? 0 : it.h0;
  const int64_t lbase = ((int64_t)it.b * a.meta.nH + lh) * a.meta.nQt;
  if (rank_out) {  // placement only: the caller supplies qt and n
    *rank_out = rank;
    it.qt = 0; it.n = 0; it.list = nullptr;
    return it;
  }
  it.qt = __ldg(a.meta.fwd_ord + lbase + rank);
  it.n = __ldg(a.meta.fwd_cnt + lbase + it.qt);
  it.list = a.meta.fwd_lst + (lbase + it.qt) * a.meta.nKt;
  return it;
}

// The item of a queue entry (index, query tile, key tiles): placement by
// arithmetic, no metadata loads.
__device__ __forceinline__ FwdItem fwd_item_queued(const FwdArgs& a, int hpc, int hb, int4 q) {
  int rank = 0;
  FwdItem it = fwd_item(a, hpc, hb, q.x, &rank);
  const int lh = a.meta.nH == 1 ? 0 : it.h0;
  const int64_t lbase = ((int64_t)it.b * a.meta.nH + lh) * a.meta.nQt;
  it.qt = q.y;
  it.n = q.z;
  it.list = a.meta.fwd_lst + (lbase + it.qt) * a.meta.nKt;
  return it;
}

// HPC: query heads per item (2, or 1); a template parameter so that each
// mode's loops are compiled for it alone.  F8: e4m3 Q, K and V^T tiles (tmV
// then maps V^T), kind::f8f6f4 products, e4m3 P.
template <int D, int HPC, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
           const __grid_constant__ FwdKernelArgs ka) {
  constexpr int kStages = FwdGeom<D, F8>::kStages;
  constexpr int kTileBytes = FwdGeom<D, F8>::kTileBytes;
  constexpr int kBoxes = FwdGeom<D, F8>::kBoxes;
  constexpr int kQBufs = FwdGeom<D, F8>::kQBufs;
  constexpr int kParts = FwdGeom<D, F8>::kParts;
  constexpr int kEntryBytes = FwdGeom<D, F8>::kEntryBytes;
  constexpr int kBoxesPerEntry = FwdGeom<D, F8>::kBoxesPerEntry;
  constexpr int kBoxCols = FwdGeom<D, F8>::kBoxCols;
  constexpr int kE = 2 * kParts;  // ring entries per key tile
  // With half-tile entries the ring holds one tile, so K runs a tile ahead of
  // V: entries go K(0), K(1), V(0), K(2), V(1), ..., V(last) -- the order the
  // MMA warp consumes them (S(T) before PV(T-1)) -- and K(T+1) streams in as
  // soon as S(T) frees its stages instead of after PV(T-1).
  constexpr bool kAhead = kParts == 2;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D, F8>& sm = *reinterpret_cast<FwdSmem<D, F8>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const FwdArgs& a = ka.a;
  const ProblemDev& pr = a.pr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int hpc = HPC;
  static_assert(HPC == 1 || (HPC == 2 && D <= 128), "two heads per item need two O regions");
  const int hb = ka.head_block;
  const int total = ka.total_items;
  // One head per item at D <= 128: the items alternate between the two
  // softmax warpgroups ("slots"), each with its own O in TMEM, so that one
  // slot's epilogue (O / l, the stores) overlaps the other slot's softmax.
  constexpr bool alt = hpc == 1 && D <= 128;
  constexpr int nsw = (hpc == 2 || alt) ? 2 : 1;  // active softmax warpgroups
  int32_t* gstatus = a.meta.status;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.s_full[2 + s], 1);
      mbar_init(&sm.p_full[s], 128);
      mbar_init(&sm.o_full[s], 1);
      mbar_init(&sm.o_last[s], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
    }
    mbar_init(&sm.drain, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.stg_full[s], 128);
      mbar_init(&sm.stg_free[s], 1);
    }
    for (int s = 0; s < 2; ++s)
      for (int u = 0; u < 2; ++u) mbar_init(&sm.bnd_ready[s][u], 128);
    for (int e = 0; e < kItemQ; ++e) {
      mbar_init(&sm.item_full[e], 1);
      mbar_init(&sm.item_empty[e], 1 + 4 * nsw);  // the MMA warp and every active softmax warp
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  if (warp >= 8) {
    regs_dec<FwdRegs<D, HPC, F8>::kOther>();
    if (warp == 8) {
    // ---------------------------------------------------------------- producer
    // The whole warp runs the loop (waits included); the elected lane issues.
    // Ring entries (counted across items) go K, V per key tile (K halves then
    // V halves at D = 256).  An item's Q tiles go in after its first K entry,
    // once the previous item's last S GEMM of that slot has released them.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    int t = 0, nq = 0;       // ring entries issued; items whose Q tiles were issued
    int q_issued[2] = {0, 0};  // Q loads issued per slot
    bool ok = true;
    unsigned long long* sched = a.meta.sched;
    // Next item index from the device-wide counter, or -1.  The CTA that
    // fetches the last "-1" of the launch puts the counters back to zero (no
    // CTA touches them afterwards), ready for the next call.
    auto fetch = [&]() -> int {
      unsigned long long v = 0ull;
      if (lane == 0) {
        v = atomicAdd(&sched[0], 1ull);
        if (v >= static_cast<unsigned long long>(total)) {
          __threadfence();
          if (atomicAdd(&sched[1], 1ull) == gridDim.x - 1ull) {
            atomicExch(&sched[0], 0ull);
            atomicExch(&sched[1], 0ull);
          }
        }
      }
      v = __shfl_sync(0xffffffffu, v, 0);
      return v < static_cast<unsigned long long>(total) ? static_cast<int>(v) : -1;
    };
    int published = 0;
    auto publish = [&](int idx, int qt, int nk) -> bool {
      const int e = published % kItemQ;
      if (published >= kItemQ) {
        const bool okw = mbar_wait(&sm.item_empty[e], ((published / kItemQ) - 1) & 1, abort_flag,
                                   gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, okw)) return false;
      }
      if (lane == 0) {
        sm.items[e] = make_int4(idx, qt, nk, 0);
        mbar_arrive(&sm.item_full[e]);  // release: the index is visible to whoever sees the phase
      }
      __syncwarp();
      ++published;
      return true;
    };
    // One ring entry: wait for its stage, then the TMA copies of a K or V
    // tile (or of its head-dim half `part`).
    auto load_entry = [&](const CUtensorMap* tm, int kt, int eb, int eg, int part) -> bool {
      const int stage = t % kStages, use = t / kStages;
      if (use > 0) {
        const bool okw = mbar_wait(&sm.kv_empty[stage], (use - 1) & 1, abort_flag, gstatus,
                                   LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, okw)) return false;
      }
      mbar_expect_tx_e(&sm.kv_full[stage], kEntryBytes);
      if (F8 && tm == &tmV) {
        // V^T [B][Hkv][128][keys]: the 128 keys of tile kt x all 128 head-dim rows.
        tma_load_4d_e(sm.kv[stage], tm, &sm.kv_full[stage], kt * kBN, 0, eg, eb);
      } else {
        for (int bx = 0; bx < kBoxesPerEntry; ++bx)
          tma_load_4d_e(sm.kv[stage] + bx * kHalfBytes, tm, &sm.kv_full[stage],
                        128 * part + kBoxCols * bx, eg, kt * kBN, eb);
      }
      ++t;
      return true;
    };
    // Items with an empty key list never enter the queue: the producer writes
    // their rows itself (O = 0, LSE = -inf).  Queued, they could deadlock the
    // CTA: an item's softmax waits for its last PV, which the MMA warp issues
    // when it opens the next non-empty item, and the longest-first order puts
    // empty items last, possibly more of them in a row than the queue holds.
    auto zero_item = [&](const FwdItem& x) {
      for (int s = 0; s < hpc; ++s) {
        const int h = x.h0 + s;
        for (int c = lane; c < kBM * (D / 8); c += 32) {
          const int r = c / (D / 8), ch = c % (D / 8);
          const int row = x.qt * kBM + r;
          if (row >= pr.Sq) continue;
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)x.b * a.o_sb +
                                (int64_t)row * a.o_ss + (int64_t)h * a.o_sh;
          reinterpret_cast<uint4*>(orow)[ch] = make_uint4(0u, 0u, 0u, 0u);
          if (ch == 0) a.lse[((int64_t)x.b * pr.Hq + h) * pr.Sq + row] = -INFINITY;
        }
      }
    };
    int prev_kt = -1, prev_b = 0, prev_g = 0;  // K ahead of V: the tile whose V is still to come
    int cur = fetch();
    FwdItem cur_it{};  // item `cur` (its metadata read once, here)
    if (cur >= 0) cur_it = fwd_item(a, hpc, hb, cur);
    int cur_n = cur >= 0 ? cur_it.n : 0;  // key tiles of item `cur`
    while (ok) {
      if (cur >= 0 && cur_n == 0) {  // an empty item: written here, never queued
        zero_item(cur_it);
        cur = fetch();
        if (cur >= 0) cur_it = fwd_item(a, hpc, hb, cur);
        cur_n = cur >= 0 ? cur_it.n : 0;
        continue;
      }
      if (!publish(cur, cur >= 0 ? cur_it.qt : 0, cur_n)) { ok = false; break; }
      if (cur < 0) break;
      const int nxt = fetch();
      const FwdItem it = cur_it;
      cur = nxt;
      if (nxt >= 0) {
        // Warm L2 with the next item's query rows while this item runs.
        const FwdItem nx = fwd_item(a, hpc, hb, nxt);
        cur_it = nx;
        cur_n = nx.n;
        if (nx.n > 0)
          for (int s = 0; s < hpc; ++s)
            for (int bx = 0; bx < kBoxes; ++bx)
              tma_prefetch_l2_4d_e(&tmQ, kBoxCols * bx, nx.h0 + s, nx.qt * kBM, nx.b);
      }
      if (it.n == 0) continue;
      const int g = it.h0 / pr.G;
      for (int u = 0; u < kE * it.n && ok; ++u) {
        const int j = u / kE, e = u % kE;
        const int part = e % kParts;
        const int kt_j = __ldg(it.list + j) >> 1;
        const bool is_v = e >= kParts;
        int kt = kt_j, eb = it.b, eg = g;
        bool skip = false;
        if (kAhead && is_v) {  // V of the previous tile (none before the stream's first)
          if (prev_kt < 0) skip = true;
          else { kt = prev_kt; eb = prev_b; eg = prev_g; }
        }
        if (!skip && !load_entry(is_v ? &tmV : &tmK, kt, eb, eg, part)) { ok = false; break; }
        if (kAhead && e == kE - 1) { prev_kt = kt_j; prev_b = it.b; prev_g = g; }
        if (u == 0) {
          // Two heads: buffer s holds slot s's Q for every item.  One head:
          // the two buffers alternate between items, so the next item's Q
          // never waits for this item's last S GEMM.
          for (int s = 0; s < hpc && ok; ++s) {
            const int qb = hpc == 1 ? (kQBufs == 2 ? (nq & 1) : 0) : s;
            const int quse = hpc == 1 && kQBufs == 2 ? (nq >> 1) : nq;
            if (quse > 0) {
              ok = mbar_wait(&sm.q_empty[qb], (quse - 1) & 1, abort_flag, gstatus,
                             LCATTN_ERR_DEVICE_TIMEOUT);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            }
            mbar_expect_tx_e(&sm.q_full[qb], kTileBytes);
            for (int bx = 0; bx < kBoxes; ++bx)
              tma_load_4d_e(sm.q[qb] + bx * kHalfBytes, &tmQ, &sm.q_full[qb], kBoxCols * bx, it.h0 + s,
                            it.qt * kBM, it.b);
            ++q_issued[qb];
          }
          if (!ok) break;
          ++nq;
        }
      }
    }
    // The last tile's V (K ran one tile ahead).
    if (kAhead && ok && prev_kt >= 0)
      for (int part = 0; part < kParts && ok; ++part) ok = load_entry(&tmV, prev_kt, prev_b, prev_g, part);
    // Never leave copies in flight: wait (bounded, ignoring the abort word) for
    // the last load issued on each ring stage and for the last Q tiles.
    for (int u = max(0, t - kStages); u < t; ++u) {
      int dummy = 0;
      mbar_wait(&sm.kv_full[u % kStages], (u / kStages) & 1, &dummy, gstatus,
                LCATTN_ERR_DEVICE_TIMEOUT);
    }
    for (int s = 0; s < 2; ++s) {
      if (q_issued[s] == 0) continue;
      int dummy = 0;
      mbar_wait(&sm.q_full[s], (q_issued[s] - 1) & 1, &dummy, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
    }
    } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop; every tcgen05.mma / commit is issued by one
    // elected lane (see the elected-lane forms in the primitives header).
    // The issue stream is flat over this CTA's tiles (T counts them across
    // items): step T issues PV(T-1) and S(T) per slot, so the first S of an
    // item follows the previous item's last PV without a gap.  PV(T-1) starts
    // a fresh accumulation when tile T-1 opened its item; by then the softmax
    // has read the previous item's O (it does so before releasing the item's
    // first P).
    {
      const uint32_t idesc_qk = F8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc_pv = F8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D / kParts, false, true);
      // Base descriptors; stage s of the ring is kTileBytes further on.
      const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dq1 = sdesc_sw128(smem_u32(sm.q[kQBufs - 1]), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(sm.kv[0]), 16, 1024);          // K tile, K-major
      // V tile read MN-major (bf16), or V^T tile read K-major (e4m3).
      const uint64_t dv0 = sdesc_sw128(smem_u32(sm.kv[0]), F8 ? 16u : static_cast<uint32_t>(kHalfBytes), 1024);
      // S (+)= Q K^T over one ring entry: k-steps of 32 bytes inside the
      // 128-byte swizzled rows, the next 64-column box after four of them.
      auto gemm_s = [&](uint32_t tS, uint64_t qp, uint64_t kb, bool first) {
        if constexpr (F8) {
          if (first) mma8_ss_e<0>(tS, qp, kb, idesc_qk);
          else mma8_ss_e<1>(tS, qp, kb, idesc_qk);
        } else {
          if (first) mma_ss_e<0>(tS, qp, kb, idesc_qk);
          else mma_ss_e<1>(tS, qp, kb, idesc_qk);
        }
        #pragma unroll
        for (int kk = 1; kk < FwdGeom<D, F8>::kSSteps; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          if constexpr (F8) mma8_ss_e<1>(tS, sdesc_add(qp, off), sdesc_add(kb, off), idesc_qk);
          else mma_ss_e<1>(tS, sdesc_add(qp, off), sdesc_add(kb, off), idesc_qk);
        }
      };
      // O (+)= P V: A = P from TMEM (8 columns per k-step: 16 bf16 or 32 e4m3
      // keys), B = V read MN-major (16 key rows, 2048 bytes, per k-step) or V^T
      // read K-major (32 keys, 32 bytes, per k-step).
      auto gemm_pv = [&](uint32_t tO, uint32_t tP, uint64_t vb, uint32_t acc) {
        if constexpr (F8) {
          mma8_ts_er(tO, tP, vb, idesc_pv, acc);
          #pragma unroll
          for (int kk = 1; kk < FwdGeom<D, F8>::kPvSteps; ++kk)
            mma8_ts_er(tO, tP + kk * 8, sdesc_add(vb, kk * 32), idesc_pv, 1u);
        } else {
          mma_ts_er(tO, tP, vb, idesc_pv, acc);
          #pragma unroll
          for (int kk = 1; kk < FwdGeom<D, F8>::kPvSteps; ++kk)
            mma_ts_e<1>(tO, tP + kk * 8, sdesc_add(vb, kk * 2048), idesc_pv);
        }
      };
      bool ok = true;
      int T = 0, nq = 0;
      uint32_t pv_acc = 0u;  // accumulate flag of the pending PV(T-1)
      auto issue_pv = [&](int s, bool last) -> bool {
        const uint32_t tS = tmem + s * 128, tO = tmem + 256 + s * 128;
        const bool okw = mbar_wait(&sm.p_full[s], (T - 1) & 1, abort_flag, gstatus,
                                   LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, okw)) return false;
        tc_fence_after();
        const int tv = 2 * T - 1;
        const uint64_t vb = sdesc_add(dv0, (tv % kStages) * kTileBytes);
        gemm_pv(tO, tS, vb, pv_acc);  // O += P V
        tc_commit_e(&sm.o_full[s]);
        if (last) tc_commit_e(&sm.o_last[s]);  // the item's O is complete
        return true;
      };
      if (hpc == 1) {
        // One head per item: S is double-buffered in the two S regions, and
        // S(t) is issued before PV(t-1), so the softmax of tile t-1 overlaps
        // S(t) and finds S(t) done when it finishes.  S(t) overwrites the
        // buffer of P(t-2), which PV(t-2), issued before it, has read.  With
        // alternating slots, the item's slot (its Q buffer) picks the O region
        // and the S barriers.
        uint32_t acc_prev = 0u;
        int prev_slot = 0;  // slot of the item of tile T-1
        auto issue_pv1 = [&](int tt, uint32_t acc, bool last, bool stream_last, int ps) -> bool {
          // P(tt) is released on the barrier of its S buffer: one barrier per
          // buffer keeps the softmax (which can run a tile ahead) from
          // completing a second phase before this wait has seen the first.
          bool okw = mbar_wait(&sm.p_full[tt & 1], (tt >> 1) & 1, abort_flag, gstatus,
                               LCATTN_ERR_DEVICE_TIMEOUT);
          const uint32_t tP = tmem + (tt & 1) * 128;
          #pragma unroll 1
          for (int part = 0; part < kParts; ++part) {
            // V entry of tile tt: columns [part * D/kParts, ...) of O.
            const int tv = !kAhead || stream_last ? kE * tt + kParts + part : kE * tt + kE + part;
            if (okw) okw = mbar_wait(&sm.kv_full[tv % kStages], (tv / kStages) & 1, abort_flag, gstatus,
                                     LCATTN_ERR_DEVICE_TIMEOUT);
            if (!__all_sync(0xffffffffu, okw)) return false;
            tc_fence_after();
            const uint64_t vb = sdesc_add(dv0, (tv % kStages) * kEntryBytes);
            const uint32_t tOp = tmem + 256 + ps * 128 + part * (D / kParts);
            gemm_pv(tOp, tP, vb, acc);
            tc_commit_e(&sm.kv_empty[tv % kStages]);
          }
          tc_commit_e(&sm.o_full[ps]);
          if (last) tc_commit_e(&sm.o_last[ps]);  // the item's O is complete
          return true;
        };
        for (int k = 0; ok; ++k) {
          const int e = k % kItemQ;
          ok = mbar_wait(&sm.item_full[e], (k / kItemQ) & 1, abort_flag, gstatus,
                         LCATTN_ERR_DEVICE_TIMEOUT);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          const int4 iq = sm.items[e];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.item_empty[e]);
          if (iq.x < 0) break;
          const int n = iq.z;
          if (n == 0) continue;
          const int qb = kQBufs == 2 ? (nq & 1) : 0;
          const int quse = kQBufs == 2 ? (nq >> 1) : nq;
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full[qb], quse & 1, abort_flag, gstatus,
                                                 LCATTN_ERR_DEVICE_TIMEOUT));
          if (!ok) break;
          const uint64_t qd = qb ? dq1 : dq0;
          const int slot = alt ? qb : 0;
          for (int j = 0; j < n; ++j, ++T) {
            const uint32_t tS = tmem + (T & 1) * 128;
            #pragma unroll 1
            for (int part = 0; part < kParts; ++part) {  // K entries: head-dim parts of the tile
              const int tk = !kAhead ? kE * T + part : (T == 0 ? part : kE * T - kParts + part);
              ok = __all_sync(0xffffffffu, mbar_wait(&sm.kv_full[tk % kStages], (tk / kStages) & 1,
                                                     abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT));
              if (!ok) break;
              tc_fence_after();
              const uint64_t kb = sdesc_add(dk0, (tk % kStages) * kEntryBytes);
              const uint64_t qp = sdesc_add(qd, part * kEntryBytes);
              gemm_s(tS, qp, kb, part == 0);
              tc_commit_e(&sm.kv_empty[tk % kStages]);
            }
            if (!ok) break;
            tc_commit_e(&sm.s_full[2 * slot + (T & 1)]);
            if (j == n - 1) tc_commit_e(&sm.q_empty[qb]);  // this item's Q is read for good
            // PV(T-1) closes the previous item when tile T opens a new one.
            if (T > 0 && !issue_pv1(T - 1, acc_prev, j == 0, false, prev_slot)) { ok = false; break; }
            acc_prev = j > 0 ? 1u : 0u;
            prev_slot = slot;
          }
          if (ok) ++nq;
        }
        if (ok && T > 0) issue_pv1(T - 1, acc_prev, true, true, prev_slot);
      } else if (D <= 128)  // two heads per item (never at D = 256)
      for (int k = 0; ok; ++k) {
        const int e = k % kItemQ;
        ok = mbar_wait(&sm.item_full[e], (k / kItemQ) & 1, abort_flag, gstatus,
                       LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const int4 iq = sm.items[e];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.item_empty[e]);
        if (iq.x < 0) break;
        const int n = iq.z;
        if (n == 0) continue;
        for (int j = 0; j < n; ++j, ++T) {
          const int tk = 2 * T, tv = 2 * T - 1;
          ok = mbar_wait(&sm.kv_full[tk % kStages], (tk / kStages) & 1, abort_flag, gstatus,
                         LCATTN_ERR_DEVICE_TIMEOUT);
          if (ok && T > 0)
            ok = mbar_wait(&sm.kv_full[tv % kStages], (tv / kStages) & 1, abort_flag, gstatus,
                           LCATTN_ERR_DEVICE_TIMEOUT);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kb = sdesc_add(dk0, (tk % kStages) * kTileBytes);
          #pragma unroll (D == 64 ? 1 : 2)  // rolled at head dim 64, whose MMA warp spills unrolled
          for (int s = 0; s < hpc; ++s) {
            if (T > 0 && !issue_pv(s, j == 0)) { ok = false; break; }
            if (j == 0) {
              ok = mbar_wait(&sm.q_full[s], nq & 1, abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
              tc_fence_after();
            }
            // S = Q K^T, both K-major.
            const uint32_t tS = tmem + s * 128;
            const uint64_t qd = s ? dq1 : dq0;
            gemm_s(tS, qd, kb, true);
            tc_commit_e(&sm.s_full[s]);
            if (j == n - 1) tc_commit_e(&sm.q_empty[s]);  // Q of this slot is read for good
          }
          if (!ok) break;
          tc_commit_e(&sm.kv_empty[tk % kStages]);
          if (T > 0) tc_commit_e(&sm.kv_empty[tv % kStages]);
          pv_acc = j > 0 ? 1u : 0u;
        }
        if (ok) ++nq;
      }
      // The last PV of the sequence (two heads per item).
      if (hpc != 1 && ok && T > 0) {
        const int tv = 2 * T - 1;
        ok = mbar_wait(&sm.kv_full[tv % kStages], (tv / kStages) & 1, abort_flag, gstatus,
                       LCATTN_ERR_DEVICE_TIMEOUT);
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after();
          for (int s = 0; s < hpc; ++s)
            if (!issue_pv(s, true)) break;
          tc_commit_e(&sm.kv_empty[tv % kStages]);
        }
      }
      // Drain: every MMA issued above has completed once this barrier flips.
      tc_commit_e(&sm.drain);
      int dummy = 0;
      mbar_wait(&sm.drain, 0, &dummy, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
    }
    }
  } else {
    regs_inc<FwdRegs<D, HPC, F8>::kSoftmax>();
    // ---------------------------------------------------------------- softmax
    const int s = warp >> 2;
    const int r = tid & 127;  // == 32 * (warp % 4) + lane: this thread's TMEM lane
    if (s < nsw) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const uint32_t tO = tmem + lane_off + 256 + s * 128;
      const float sl2 = a.scale_log2;
      constexpr float kLog2PScale = F8 ? 4.0f : 0.0f;  // log2 of FwdGeom::kPScale
      static_assert(FwdGeom<D, F8>::kPScale == (F8 ? 16.0f : 1.0f), "P scale and its log2");
      const int last_kt = (pr.Sk - 1) / kBN;
      const bool ragged_k = (pr.Sk % kBN) != 0;
      const bool use_rows = a.mask.kind == LCATTN_MASK_COLBOUNDS && a.mask.row_bounds != nullptr;
      bool ok = true;
      int T = 0;          // tiles of this CTA processed before the current item
      int n_partial = 0;  // partial column-bounds tiles staged so far (selects the buffer)
      // Counter parities (the barrier waits need no more).  Alternating slots:
      // bit b < 2 = this slot's key tiles so far in S buffer b, bit 2 = items
      // with at least one key tile seen by either slot.  Bit 3 = this slot's
      // items with at least one key tile finished so far.  Bit 4 = epilogues
      // so far; bit 5 = the staging buffers may still be read by TMA stores.
      uint32_t pbits = 0u;
      // The staging buffers (and the column bounds that share them) are free
      // again once the last epilogue's TMA stores have read them: its issuing
      // lane waits for that and releases the buffers; every thread of the slot
      // waits for the release before writing there again.
      auto stg_reclaim = [&]() -> bool {
        if (!(pbits & 32u)) return true;
        if (warp == 4 * s && lane == 0) {
          bulk_wait_read0();
          mbar_arrive(&sm.stg_free[s]);
        }
        __syncwarp();
        const bool okw = mbar_wait(&sm.stg_free[s], ((pbits >> 4) & 1u) ^ 1u, abort_flag, gstatus,
                                   LCATTN_ERR_DEVICE_TIMEOUT);
        pbits &= ~32u;
        return __all_sync(0xffffffffu, okw);
      };
      for (int k = 0; ok; ++k) {
        const int e = k % kItemQ;
        ok = mbar_wait(&sm.item_full[e], (k / kItemQ) & 1, abort_flag, gstatus,
                       LCATTN_ERR_DEVICE_TIMEOUT);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const int4 iq = sm.items[e];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.item_empty[e]);
        if (iq.x < 0) break;
        const FwdItem it = fwd_item_queued(a, hpc, hb, iq);
        const int n = it.n, b = it.b;
        if (alt && n > 0) {
          const bool mine = static_cast<int>((pbits >> 2) & 1u) == s;
          pbits ^= 4u;
          if (!mine) { T += n; continue; }  // the other slot's item
          // Alternating slots: this slot's previous epilogue was an item ago,
          // so its stores have long read the staging buffer.
          if (!stg_reclaim()) { ok = false; break; }
        }
        const int h = it.h0 + (hpc == 2 ? s : 0);
        const int row = it.qt * kBM + r;
        int qb_row = 0;
        if (a.mask.kind == LCATTN_MASK_BLOCKMAP)
          qb_row = block_of(a.mask.q_offs, a.mask.nQb, min(row, pr.Sq - 1));
        // This row's allowed keys [c0, d0) U [c1, d1), when the descriptor carries
        // the per-row form (rows past Sq allow nothing).
        int4 rb = make_int4(0, 0, 0, 0);
        if (use_rows && row < pr.Sq) rb = __ldg(a.mask.row_bounds + (int64_t)b * pr.Sq + row);
        float m_run = -INFINITY, l_run = 0.f;
        int e_next = n > 0 ? __ldg(it.list) : 0;
        for (int j = 0; j < n; ++j) {
          const int e = e_next;
          if (j + 1 < n) e_next = __ldg(it.list + j + 1);  // prefetch the next entry
          const int kt = e >> 1;
          const bool partial = (e & 1) != 0;
          const bool masked = partial || (ragged_k && kt == last_kt);
          uint32_t mw[4];
          if (masked && partial && use_rows) {
            // The row's two key intervals, clipped to the tile's valid columns.
            const int j0 = kt * kBN, j1 = min(pr.Sk, j0 + kBN);
            const int lo0 = max(rb.x, j0) - j0, hi0 = min(rb.y, j1) - j0;
            const int lo1 = max(rb.z, j0) - j0, hi1 = min(rb.w, j1) - j0;
            #pragma unroll
            for (int w = 0; w < 4; ++w)
              mw[w] = range_bits(lo0, hi0, 32 * w) | range_bits(lo1, hi1, 32 * w);
          } else if (masked) {
            const int4* bnd = nullptr;
            if (partial && a.mask.kind == LCATTN_MASK_COLBOUNDS) {
              // Stage the tile's 128 column bounds in shared memory: one coalesced
              // load per thread instead of 128 dependent loads per thread.
              if (!alt && !stg_reclaim()) { ok = false; break; }
              const int u = n_partial & 1;
              const int key = kt * kBN + r;
              int4* bs = reinterpret_cast<int4*>(sm.stg[s]) + u * kBN;
              bs[r] = key < pr.Sk ? __ldg(a.mask.col_bounds + (int64_t)b * pr.Sk + key)
                                            : make_int4(0, 0, 0, 0);
              mbar_arrive(&sm.bnd_ready[s][u]);
              ok = mbar_wait(&sm.bnd_ready[s][u], (n_partial >> 1) & 1, abort_flag, gstatus,
                             LCATTN_ERR_DEVICE_TIMEOUT);
              if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
              bnd = bs;
              ++n_partial;
            }
            tile_mask_bits(a.mask, pr, b, h, row, qb_row, kt, partial, bnd, mw);
          }
          // Two heads: slot s's S region every tile.  One head: the two S
          // regions alternate between tiles.
          const int sb = hpc == 1 ? ((T + j) & 1) : s;
          const uint32_t tS = tmem + lane_off + sb * 128;
          // S barriers: per slot (two heads, a phase per tile), per buffer
          // (one head), per slot and buffer (alternating: a phase per tile of
          // this slot in that buffer, so a slot never waits on a phase that
          // the other slot's tiles could have run past).
          const int sfi = hpc == 2 ? s : (alt ? 2 * s + sb : sb);
          int sph;
          if (hpc == 2) sph = T + j;
          else if (alt) { sph = static_cast<int>(pbits >> sb); pbits ^= 1u << sb; }
          else sph = (T + j) >> 1;
          ok = mbar_wait(&sm.s_full[sfi], sph & 1, abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
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
            const uint32_t w0 = mw[0], w1 = mw[1], w2 = mw[2], w3 = mw[3];
            #pragma unroll
            for (int c = 0; c < 128; ++c) {
              const uint32_t w = c < 32 ? w0 : (c < 64 ? w1 : (c < 96 ? w2 : w3));
              if (!((w >> (c & 31)) & 1u)) x[c] = -INFINITY;
            }
          }
          // Row max: four independent chains of three-input maxima (two new
          // columns per instruction; one long chain would be latency bound).
          float m4[4];
          #pragma unroll
          for (int c = 0; c < 4; ++c) m4[c] = fmaxf(x[2 * c], x[2 * c + 1]);
          #pragma unroll
          for (int c = 8; c < 128; c += 2) m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], x[c], x[c + 1]);
          const float m_tile = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]) * sl2;  // -inf stays -inf
          const bool need = m_tile > m_run + FwdGeom<D, F8>::kRescaleThreshold;
          const bool warp_rescale = __any_sync(0xffffffffu, need) && j > 0;
          const float m_new = need ? m_tile : m_run;
          const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;  // exp2(-inf) = 0
          m_run = m_new;
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          // P = exp2(S * scale * log2(e) - m): the scaling and the row sum run
          // on column pairs (paired fp32 instructions), the exponentials one by one.
          // e4m3 P is P * kPScale (the shift folded into the exponent); the row
          // sum l then carries the same factor, which cancels in O / l.
          const float negm_s = -(m_use - kLog2PScale);
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
            // O holds PV up to tile j-1: wait for it, then scale it in place
            // before PV(j) is issued (which needs p_full below).
            // PV(j-1) of this item: phase (slot's tiles so far) - 2, whose
            // parity is that of the slot's tile count (bits 0 and 1).
            const int oph = alt ? static_cast<int>(pbits ^ (pbits >> 1)) : (T + j - 1);
            ok = mbar_wait(&sm.o_full[s], oph & 1, abort_flag, gstatus, LCATTN_ERR_DEVICE_TIMEOUT);
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
        // ---- epilogue: O / l and LSE.  O is read (and the read waited for)
        // before the next item's first P is released, which is what lets the
        // next item's first PV overwrite it.  The wait is on the per-item
        // barrier: with S issued ahead (one head per item) the softmax can
        // finish an item while two of its PVs are still pending, and a parity
        // wait on the per-PV barrier could then match an older phase.
        bool have_o = ok && n > 0;
        if (have_o) {
          have_o = mbar_wait(&sm.o_last[s], (pbits >> 3) & 1, abort_flag, gstatus,
                             LCATTN_ERR_DEVICE_TIMEOUT);
          have_o = __all_sync(0xffffffffu, have_o);
          tc_fence_after();
        }
        if (!alt && ok && (have_o || n == 0) && !stg_reclaim()) ok = false;
        if (ok && (have_o || n == 0)) {
          const bool live = l_run > 0.f;
          const float inv = live ? a.o_scale / l_run : 0.f;
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.o_sb +
                                (int64_t)row * a.o_ss + (int64_t)h * a.o_sh;
          // The first kTmaCols columns go out through shared memory and TMA
          // stores (one 64-column box per slot; two with one slot), the rest
          // as 32-byte stores from the registers, one row per thread.
          constexpr int kTmaCols = nsw == 2 ? 64 : (D < 128 ? D : 128);
          // All of O in one round trip when it fits the registers (D <= 128),
          // else 32 columns at a time; then O / l on column pairs.
          constexpr int kBatch = D <= 128 ? D : 32;
          const float2 inv2 = make_float2(inv, inv);
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
          #pragma unroll
          for (int c = 0; c < kBatch / 32; ++c) {
            uint32_t pk[16];
            #pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 y = mul2(make_float2(__uint_as_float(o32[c * 32 + 2 * i]),
                                                __uint_as_float(o32[c * 32 + 2 * i + 1])), inv2);
              pk[i] = pack_bf16x2(y.x, y.y);
            }
            const int cc = c0 + c * 32;
            if (cc < kTmaCols) {
              // Row r of a 128-byte-swizzled box: 16-byte chunk j sits at j ^ (r % 8).
              uint8_t* srow = sm.stg[nsw == 2 ? s : (cc >> 6)] + r * 128;
              const int j0 = (cc & 63) >> 3;
              #pragma unroll
              for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(srow + (((j0 + i) ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
              if (cc + 32 == kTmaCols) {
                fence_proxy_async_smem();
                mbar_arrive(&sm.stg_full[s]);
                if (warp == 4 * s) {
                  const bool okf = __all_sync(0xffffffffu,
                                              mbar_wait(&sm.stg_full[s], (pbits >> 4) & 1u, abort_flag,
                                                        gstatus, LCATTN_ERR_DEVICE_TIMEOUT));
                  if (okf && lane == 0) {
                    #pragma unroll
                    for (int bx = 0; bx < kTmaCols / 64; ++bx)
                      tma_store_4d(&tmO, sm.stg[nsw == 2 ? s : bx], 64 * bx, h, it.qt * kBM, b);
                    bulk_commit();
                  }
                  __syncwarp();
                  if (!okf) ok = false;
                }
                pbits |= 32u;
              }
            } else if (row < pr.Sq) {
              __nv_bfloat16* dst = orow + cc;
              if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
                st_global_v8(dst, pk);
                st_global_v8(dst + 16, pk + 8);
              } else {
                #pragma unroll
                for (int i = 0; i < 4; ++i)
                  reinterpret_cast<uint4*>(dst)[i] =
                      make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
              }
            }
          }
          }
          pbits ^= 16u;
          if (row < pr.Sq)
            a.lse[((int64_t)b * pr.Hq + h) * pr.Sq + row] =
                live ? (m_run - kLog2PScale + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        }
        if (n > 0 && !have_o) ok = false;
        if (n > 0) pbits ^= 8u;
        T += n;
      }
      // The shared memory goes away with the CTA: the last TMA stores must
      // have read it (their global writes complete with the grid).
      if (warp == 4 * s && lane == 0) bulk_wait_read0();
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

template <int D, int HPC, bool F8>
cudaError_t launch_fwd_mode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const FwdKernelArgs& ka, int grid, cudaStream_t st) {
  static bool attr_done = false;
  const size_t smem = sizeof(FwdSmem<D, F8>) + 1024;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, HPC, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  fwd_kernel<D, HPC, F8><<<(unsigned)grid, kThreads, smem, st>>>(tq, tk, tv, to, ka);
  return cudaGetLastError();
}

template <int D, bool F8 = false>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdArgs& a, cudaStream_t st) {
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  FwdKernelArgs ka;
  ka.a = a;
  // Two query heads per CTA when they share the key tiles and the tile list
  // (and two 256-column O accumulators would not fit in TMEM at D = 256).
  ka.heads_per_cta = (D <= 128 && a.meta.nH == 1 && a.pr.G % 2 == 0) ? 2 : 1;
  // One head per item: the smallest block of whole GQA groups (a divisor of Hq)
  // whose items fill the GPU twice over.
  ka.head_block = a.pr.Hq;
  for (int d = a.pr.G; d <= a.pr.Hq; d += a.pr.G)
    if (a.pr.Hq % d == 0 && (int64_t)d * a.meta.nQt >= 2 * (int64_t)nsm) { ka.head_block = d; break; }
  const int64_t total = (int64_t)(a.pr.Hq / ka.heads_per_cta) * a.pr.B * a.meta.nQt;
  if (total > 0x7fffffffLL) return cudaErrorInvalidValue;  // far beyond any problem that fits in memory
  ka.total_items = static_cast<int>(total);
  // Persistent: one CTA per SM (shared memory admits one), never more CTAs than items.
  const int grid = ka.total_items < nsm ? ka.total_items : nsm;
  if constexpr (D <= 128)
    if (ka.heads_per_cta == 2) return launch_fwd_mode<D, 2, F8>(tq, tk, tv, to, ka, grid, st);
  return launch_fwd_mode<D, 1, F8>(tq, tk, tv, to, ka, grid, st);
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& a, cudaStream_t st) {
  if (a.pr.D == 64) return launch_fwd_d<64>(tq, tk, tv, to, a, st);
  if (a.pr.D == 256) return launch_fwd_d<256>(tq, tk, tv, to, a, st);
  return launch_fwd_d<128>(tq, tk, tv, to, a, st);
}

cudaError_t launch_fwd_e4m3(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                            const CUtensorMap& to, const FwdArgs& a, cudaStream_t st) {
  if (a.pr.D != 128) return cudaErrorInvalidValue;
  return launch_fwd_d<128, true>(tq, tk, tvt, to, a, st);
}

}  // namespace lcattn
