// Mask compiler: tile classification, compacted tile lists and longest-first
// orders (the step that lets the attention kernels skip masked-out tiles and
// run full tiles without any per-element mask).
//
// The pages credit FlashMask's column-wise mask representation with making
// heterogeneous masks efficient ("Long-Context Attention Benchmark", xllm-io
// blog review, sections "掩码支持" and "关键洞察"); the descriptor here carries the
// allowed query rows of every key column as two intervals, and this compiler
// reduces it once per 128x128 tile to EMPTY / FULL / PARTIAL.
#include "lcattn_internal.cuh"

namespace lcattn {
namespace {

__device__ __forceinline__ int ilen(int a, int b, int r0, int r1) {
  const int lo = max(a, r0), hi = min(b, r1);
  return hi > lo ? hi - lo : 0;
}

// Largest idx in [0, n) with offs[idx] <= x (offs nondecreasing, offs[0] <= x).
__device__ __forceinline__ int block_of(const int32_t* offs, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Checks that block offsets run nondecreasing from 0 to S (one CTA; each
// thread checks a strided share of the adjacent pairs).
__global__ void validate_offsets_kernel(MaskDev m, int Sq, int Sk, int32_t* status) {
  bool ok = true;
  if (threadIdx.x == 0)
    ok = m.nQb > 0 && m.nKb > 0 && m.q_offs[0] == 0 && m.k_offs[0] == 0 &&
         m.q_offs[m.nQb] == Sq && m.k_offs[m.nKb] == Sk;
  for (int i = threadIdx.x; i < m.nQb; i += blockDim.x) ok &= __ldg(m.q_offs + i) <= __ldg(m.q_offs + i + 1);
  for (int i = threadIdx.x; i < m.nKb; i += blockDim.x) ok &= __ldg(m.k_offs + i) <= __ldg(m.k_offs + i + 1);
  if (!__syncthreads_and(ok) && threadIdx.x == 0) atomicCAS(status, 0, LCATTN_ERR_DEVICE_MASK);
}

// Column bounds, one warp per tile: count the allowed rows of each column
// inside the tile's row range (union of the two intervals) and compare the sum
// with the tile's in-range area.
__global__ void classify_kernel(ProblemDev pr, MaskDev m, TileMetaDev t) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t total = (int64_t)t.B * t.nH * t.nQt * t.nKt;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
       w += warps_total) {
    const int kt = (int)(w % t.nKt);
    const int qt = (int)((w / t.nKt) % t.nQt);
    const int b = (int)(w / ((int64_t)t.nKt * t.nQt * t.nH));
    const int r0 = qt * kBM, r1 = min(pr.Sq, r0 + kBM);
    const int c0 = kt * kBN, c1 = min(pr.Sk, c0 + kBN);
    int cnt = 0;
    const int4* cb = m.col_bounds + (int64_t)b * pr.Sk;
    for (int j = c0 + lane; j < c1; j += 32) {
      const int4 v = __ldg(cb + j);
      cnt += ilen(v.x, v.y, r0, r1) + ilen(v.z, v.w, r0, r1) -
             ilen(max(v.x, v.z), min(v.y, v.w), r0, r1);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    const int area = (r1 - r0) * (c1 - c0);
    const uint8_t cls =
        cnt == 0 ? LCATTN_TILE_EMPTY : (cnt == area ? LCATTN_TILE_FULL : LCATTN_TILE_PARTIAL);
    if (lane == 0) t.cls[w] = cls;
  }
}

// Block maps: one warp per row of tiles (batch, head, query tile); lanes take
// key tiles.  The query-block range is found once per row; each lane looks up
// its tile's key-block range and scans the covered (query block, key block)
// pairs.
__global__ void classify_blockmap_kernel(ProblemDev pr, MaskDev m, TileMetaDev t) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t rows = (int64_t)t.B * t.nH * t.nQt;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows;
       w += warps_total) {
    const int qt = (int)(w % t.nQt);
    const int h = (int)((w / t.nQt) % t.nH);
    const int b = (int)(w / ((int64_t)t.nQt * t.nH));
    const int r0 = qt * kBM, r1 = min(pr.Sq, r0 + kBM);
    const int qb0 = block_of(m.q_offs, m.nQb, r0), qb1 = block_of(m.q_offs, m.nQb, r1 - 1);
    const uint8_t* map = m.block_map + (((int64_t)b * pr.Hq + h) * m.nQb) * m.nKb;
    uint8_t* out = t.cls + w * t.nKt;
    for (int kt = lane; kt < t.nKt; kt += 32) {
      const int c0 = kt * kBN, c1 = min(pr.Sk, c0 + kBN);
      const int kb0 = block_of(m.k_offs, m.nKb, c0), kb1 = block_of(m.k_offs, m.nKb, c1 - 1);
      bool any_keep = false, any_drop = false;
      for (int qb = qb0; qb <= qb1; ++qb) {
        const int qlen = min(__ldg(m.q_offs + qb + 1), r1) - max(__ldg(m.q_offs + qb), r0);
        if (qlen <= 0) continue;
        for (int kb = kb0; kb <= kb1; ++kb) {
          const int klen = min(__ldg(m.k_offs + kb + 1), c1) - max(__ldg(m.k_offs + kb), c0);
          if (klen <= 0) continue;
          if (__ldg(map + (int64_t)qb * m.nKb + kb)) any_keep = true; else any_drop = true;
        }
      }
      out[kt] = !any_keep ? LCATTN_TILE_EMPTY : (any_drop ? LCATTN_TILE_PARTIAL : LCATTN_TILE_FULL);
    }
  }
}

// Backward lists (fixed key tile) through a 32 x 32 shared-memory transpose of
// the class bytes: the block reads 32 query-tile rows x 32 key tiles at a time
// (row-contiguous), and warp c compacts key tile kt0 + c over those rows.
__global__ void __launch_bounds__(1024) bwd_list_kernel(TileMetaDev t) {
  __shared__ uint8_t tile[32][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nChunks = (t.nKt + 31) / 32;
  const int64_t bh = blockIdx.x / nChunks;
  const int kt0 = (int)(blockIdx.x % nChunks) * 32;
  const uint8_t* cls = t.cls + bh * t.nQt * t.nKt;
  const int kt = kt0 + warp;
  int32_t* lst = t.bwd_lst + (bh * t.nKt + kt) * t.nQt;
  int n = 0;
  for (int qt0 = 0; qt0 < t.nQt; qt0 += 32) {
    const int qr = qt0 + warp, kc = kt0 + lane;
    tile[warp][lane] = (qr < t.nQt && kc < t.nKt) ? cls[(int64_t)qr * t.nKt + kc] : (uint8_t)LCATTN_TILE_EMPTY;
    __syncthreads();
    const uint8_t c = tile[lane][warp];  // row qt0 + lane, key tile kt
    const unsigned bal = __ballot_sync(0xffffffffu, c != LCATTN_TILE_EMPTY);
    if (kt < t.nKt && c != LCATTN_TILE_EMPTY)
      lst[n + __popc(bal & ((1u << lane) - 1u))] = ((qt0 + lane) << 1) | (c == LCATTN_TILE_PARTIAL ? 1 : 0);
    n += __popc(bal);
    __syncthreads();
  }
  if (lane == 0 && kt < t.nKt) t.bwd_cnt[bh * t.nKt + kt] = n;
}

// One warp per row of tiles (forward: fixed query tile) or column of tiles
// (backward: fixed key tile); non-empty entries are compacted in order with a
// ballot prefix.
template <bool kByQuery>
__global__ void list_kernel(TileMetaDev t) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int nOuter = kByQuery ? t.nQt : t.nKt;
  const int nInner = kByQuery ? t.nKt : t.nQt;
  const int64_t total = (int64_t)t.B * t.nH * nOuter;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
       w += warps_total) {
    const int outer = (int)(w % nOuter);
    const int64_t bh = w / nOuter;
    const uint8_t* cls = t.cls + bh * t.nQt * t.nKt;
    int32_t* lst = (kByQuery ? t.fwd_lst : t.bwd_lst) + w * nInner;
    int n = 0;
    for (int i0 = 0; i0 < nInner; i0 += 32) {
      const int i = i0 + lane;
      uint8_t c = LCATTN_TILE_EMPTY;
      if (i < nInner) c = kByQuery ? cls[(int64_t)outer * t.nKt + i] : cls[(int64_t)i * t.nKt + outer];
      const unsigned bal = __ballot_sync(0xffffffffu, c != LCATTN_TILE_EMPTY);
      if (c != LCATTN_TILE_EMPTY)
        lst[n + __popc(bal & ((1u << lane) - 1u))] = (i << 1) | (c == LCATTN_TILE_PARTIAL ? 1 : 0);
      n += __popc(bal);
    }
    if (lane == 0) (kByQuery ? t.fwd_cnt : t.bwd_cnt)[w] = n;
  }
}

// Longest-first order of the tiles of one (batch, list head): item i goes to
// rank #{j : cnt[j] > cnt[i]} + #{j < i : cnt[j] == cnt[i]} (stable).
template <bool kByQuery>
__global__ void order_kernel(TileMetaDev t) {
  extern __shared__ int32_t cnt_s[];
  const int n = kByQuery ? t.nQt : t.nKt;
  const int64_t bh = blockIdx.x;
  const int32_t* cnt = (kByQuery ? t.fwd_cnt : t.bwd_cnt) + bh * n;
  int32_t* ord = (kByQuery ? t.fwd_ord : t.bwd_ord) + bh * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) cnt_s[i] = cnt[i];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int ci = cnt_s[i];
    int r = 0;
    for (int j = 0; j < n; ++j) {
      const int cj = cnt_s[j];
      r += (cj > ci) || (cj == ci && j < i);
    }
    ord[r] = i;
  }
}

}  // namespace

cudaError_t launch_mask_compile(const ProblemDev& pr, const MaskDev& m, const TileMetaDev& t,
                                cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(t.status, 0, 32, st);  // status and scheduler words
  if (e != cudaSuccess) return e;
  if (m.kind == LCATTN_MASK_BLOCKMAP) {
    validate_offsets_kernel<<<1, 512, 0, st>>>(m, pr.Sq, pr.Sk, t.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  const int64_t tiles = (int64_t)t.B * t.nH * t.nQt * t.nKt;
  int64_t blocks = (tiles + 7) / 8;
  const int64_t cap = (int64_t)nsm * 16;
  if (blocks > cap) blocks = cap;
  if (m.kind == LCATTN_MASK_BLOCKMAP) {
    const int64_t rows = (int64_t)t.B * t.nH * t.nQt;
    int64_t rblocks = (rows + 7) / 8;
    if (rblocks > cap) rblocks = cap;
    classify_blockmap_kernel<<<(unsigned)rblocks, threads, 0, st>>>(pr, m, t);
  } else {
    classify_kernel<<<(unsigned)blocks, threads, 0, st>>>(pr, m, t);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  int64_t rows = (int64_t)t.B * t.nH * t.nQt;
  list_kernel<true><<<(unsigned)((rows + 7) / 8), threads, 0, st>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t col_blocks = (int64_t)t.B * t.nH * ((t.nKt + 31) / 32);
  bwd_list_kernel<<<(unsigned)col_blocks, 1024, 0, st>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const unsigned nbh = (unsigned)(t.B * t.nH);
  order_kernel<true><<<nbh, 1024, t.nQt * sizeof(int32_t), st>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  order_kernel<false><<<nbh, 1024, t.nKt * sizeof(int32_t), st>>>(t);
  return cudaGetLastError();
}

}  // namespace lcattn
