// Backward masked attention for sm_103a, in three launches:
//   1. pre-pass: D_i = <dO_i, O_i> (fp32) and zero the fp32 dQ accumulator;
//   2. dK/dV: one CTA per (key tile, KV head, batch).  For every query head of
//      the GQA group and every non-empty query tile of its list it recomputes
//      S^T = K Q^T and P^T = exp(S^T - LSE), forms dP^T = V dO^T and
//      dS^T = scale * P^T (dP^T - D), accumulates dV += P^T dO and
//      dK += dS^T Q in TMEM, and adds the partial dQ^T = K^T dS^T into the fp32
//      accumulator;
//   3. dQ conversion to bf16.
// The pages single the backward out as the main bottleneck of masked and
// sparse attention ("Long-Context Attention Benchmark", xllm-io blog review,
// sections "稀疏内核性能" and "核心发现总结"); the gradients are the textbook ones
// for L = <O, dO>.
//
// dK/dV kernel roles (512 threads, 4 warpgroups):
//   warps 0-3, 4-7  two warpgroups, one per half of the 128 query columns of a
//              tile.  Thread r is key row r of S^T / dP^T (TMEM lane r): it
//              builds its half of P'^T = scale * P^T and dS^T, writes both to
//              TMEM (bf16, in columns only its own warpgroup reads) and dS^T to
//              shared memory for the dQ product.  At the end warpgroup 0 stores
//              dV (= sum P'^T dO / scale), warpgroup 1 dK.
//   warps 8-11 dQ drain.  Thread r is head-dim row r of dQ^T = K^T dS^T: it
//              reads all 128 query columns out of TMEM (freeing them for the
//              next dP^T at once), then adds them into the fp32 accumulator;
//              a warp's 32 lanes cover 128 contiguous bytes of one query row,
//              one L2 request per instruction, off the MMA's critical path.
//   warp  12   producer: K, V once; Q_i, dO_i by TMA and LSE_i, D_i by plain
//              loads into a 2-deep ring.
//   warp  13   TMEM owner and MMA issuer; warps 14-15 idle (they complete the
//              warpgroup for setmaxnreg).
// TMEM: [0,128) S^T then P^T | [128,256) dP^T then dS^T, then dQ^T |
//       [256,384) dV | [384,512) dK.  At D = 64, dV and dK take 64 columns
//       each ([256,320), [320,384)) and dQ^T gets [384,512) of its own, so the
//       next dP^T does not wait for the drain.
#include <cuda_bf16.h>

#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

using namespace dev;

// Head dim D (64 or 128) is a template parameter.  Q, dO and V tiles are 128
// rows x D bf16 (D/64 boxes of 64 columns).  The K buffer is always two
// 64-column halves: with D = 64 its second half stays zero, so that the
// dQ^T = K^T dS^T product keeps M = 128 (head-dim rows 64-127 come out zero
// and are not drained).
constexpr int kHalfBytes = 16384;
template <int D> struct BwdGeom {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kBoxes = D / 64;
};
constexpr int kThreadsDkdv = 512;      // 4 warpgroups
// Register split for dK/dV (launch: 512 threads x 128): the two elementwise
// warpgroups 128 each, the dQ drain 144 (a whole dQ^T row in registers, plus
// the item state it keeps across the reductions), producer/MMA warpgroup 112.
// At head dim 64 with the dQ product the drain takes 152 and producer/MMA 104.
// Measured against 128 / 136 / 120 (same-box A/B): dK/dV 1-2% faster at head
// dim 128 and 8% at 64, with most of the drain's spills gone.
constexpr int kRegsWork = 128;
template <int D, bool kDq> struct BwdRegs {
  static constexpr int kDrain = (D == 64 && kDq) ? 152 : 144;
  static constexpr int kCtl = (D == 64 && kDq) ? 104 : 112;
  static_assert(128 * (2 * kRegsWork + kDrain + kCtl) <= kThreadsDkdv * 128, "register split");
};
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// 1. D pre-pass
// ---------------------------------------------------------------------------
template <int D>
__global__ void prepass_kernel(BwdArgs a) {
  constexpr int kPer = D / 32;  // head-dim elements per lane
  const int lane = threadIdx.x & 31;
  const int64_t nrows = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < nrows;
       w += wstride) {
    const int h = (int)(w % a.pr.Hq);
    const int i = (int)((w / a.pr.Hq) % a.pr.Sq);
    const int b = (int)(w / ((int64_t)a.pr.Hq * a.pr.Sq));
    const int64_t off = (int64_t)b * a.o_sb + (int64_t)i * a.o_ss + (int64_t)h * a.o_sh + lane * kPer;
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(
        reinterpret_cast<const __nv_bfloat16*>(a.o) + off);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(
        reinterpret_cast<const __nv_bfloat16*>(a.d_o) + off);
    float acc = 0.f;
    #pragma unroll
    for (int k = 0; k < kPer / 2; ++k) {
      const float2 of = __bfloat1622float2(__ldg(o2 + k));
      const float2 df = __bfloat1622float2(__ldg(d2 + k));
      acc = fmaf(of.x, df.x, acc);
      acc = fmaf(of.y, df.y, acc);
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.dvec[((int64_t)b * a.pr.Hq + h) * a.pr.Sq + i] = acc;
    if (a.accum || a.dq_sep) continue;  // the caller's accumulator keeps its contents / no accumulator
    float* dq = a.dq_acc + (int64_t)b * a.dqa_sb + (int64_t)i * a.dqa_ss + (int64_t)h * a.dqa_sh + lane * kPer;
    #pragma unroll
    for (int k = 0; k < kPer; k += 2) *reinterpret_cast<float2*>(dq + k) = make_float2(0.f, 0.f);
  }
  // Chunked units reduce-add dK and dV into an fp32 accumulator: clear it.
  if (a.nchunks > 1 && !a.accum) {
    const int64_t n4 = 2 * (int64_t)a.pr.B * a.pr.Sk * a.pr.Hkv * D / 4;
    float4* z = reinterpret_cast<float4*>(a.dkv_part);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4; t += (int64_t)gridDim.x * blockDim.x)
      z[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------------------
// 3. dQ conversion
// ---------------------------------------------------------------------------
template <int D>
__global__ void dq_convert_kernel(BwdArgs a) {
  const int64_t nvec = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq * (D / 8);
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(v % (D / 8));
    const int64_t row = v / (D / 8);  // (b, i, h)
    const int h = (int)(row % a.pr.Hq);
    const int i = (int)((row / a.pr.Hq) % a.pr.Sq);
    const int b = (int)(row / ((int64_t)a.pr.Hq * a.pr.Sq));
    const float4* src = reinterpret_cast<const float4*>(a.dq_acc + (int64_t)b * a.dqa_sb + (int64_t)i * a.dqa_ss +
                                                        (int64_t)h * a.dqa_sh + c * 8);
    const float4 x = src[0], y = src[1];
    uint4 out;
    out.x = pack_bf16x2(x.x, x.y);
    out.y = pack_bf16x2(x.z, x.w);
    out.z = pack_bf16x2(y.x, y.y);
    out.w = pack_bf16x2(y.z, y.w);
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.dq) + (int64_t)b * a.q_sb +
                         (int64_t)i * a.q_ss + (int64_t)h * a.q_sh + c * 8;
    *reinterpret_cast<uint4*>(dst) = out;
  }
}

// Sum of the split units' fp32 partials -> bf16 dK, dV (8 head dims per step).
template <int D>
__global__ void dkv_reduce_kernel(BwdArgs a) {
  const int64_t per = (int64_t)a.pr.B * a.pr.Sk * a.pr.Hkv * (D / 8);  // 8-wide groups per tensor
  const int64_t stride_part = 2 * (int64_t)a.pr.B * a.pr.Sk * a.pr.Hkv * D;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < 2 * per;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int w = (int)(v / per);  // 0 = dV, 1 = dK
    const int64_t r = v - (int64_t)w * per;
    const int c = (int)(r % (D / 8));
    const int64_t row = r / (D / 8);  // (b, key, g)
    const int g = (int)(row % a.pr.Hkv);
    const int key = (int)((row / a.pr.Hkv) % a.pr.Sk);
    const int b = (int)(row / ((int64_t)a.pr.Hkv * a.pr.Sk));
    const float* src = a.dkv_part + ((int64_t)w * a.pr.B * a.pr.Sk * a.pr.Hkv + row) * D + c * 8;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
    for (int p = 0; p < a.red_parts; ++p) {
      const float4 x0 = reinterpret_cast<const float4*>(src + p * stride_part)[0];
      const float4 x1 = reinterpret_cast<const float4*>(src + p * stride_part)[1];
      s0.x += x0.x; s0.y += x0.y; s0.z += x0.z; s0.w += x0.w;
      s1.x += x1.x; s1.y += x1.y; s1.z += x1.z; s1.w += x1.w;
    }
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(w == 0 ? a.dv : a.dk) +
                         (int64_t)b * (w == 0 ? a.v_sb : a.k_sb) +
                         (int64_t)key * (w == 0 ? a.v_ss : a.k_ss) +
                         (int64_t)g * (w == 0 ? a.v_sh : a.k_sh) + c * 8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(s0.x, s0.y), pack_bf16x2(s0.z, s0.w),
                                                pack_bf16x2(s1.x, s1.y), pack_bf16x2(s1.z, s1.w));
  }
}

// ---------------------------------------------------------------------------
// 2. dK / dV
// ---------------------------------------------------------------------------
template <int D>
struct BwdSmem {
  static constexpr int kTileBytes = BwdGeom<D>::kTileBytes;
  alignas(1024) uint8_t k[2 * kHalfBytes];  // second half zero when D = 64
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t dO[2][kTileBytes];
  alignas(1024) uint8_t ds[2 * kHalfBytes];  // dS^T, keys x queries, read MN-major by dQ^T
  // Stored negated, so that the paired fp32 instructions take them as plain
  // addends: -(LSE*log2(e) - log2(scale)) (-inf where P must be 0) and -D.
  alignas(16) float lse2[2][128];
  alignas(16) float dvec_s[2][128];
  uint64_t kv_full;
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, dq_free, done;
  uint32_t tmem_base;
  int abort_flag;
};

// Head dim 256: a unit is (key tile, KV head, head-dim half hd).  S^T and dP^T
// need the whole head dim, so K and V stay resident (64 KB each) and the Q and
// dO tiles stream through a 2-stage ring of 128-column halves (32 KB); the
// unit's own half of a Q or dO tile is loaded a second time for dK and dV, so
// that the ring is consumed strictly in order.  TMEM is laid out as at
// D = 128: dV and dK of the own half take 128 columns each.  227 KB in all.
template <>
struct BwdSmem<256> {
  alignas(1024) uint8_t k[4 * kHalfBytes];
  alignas(1024) uint8_t v[4 * kHalfBytes];
  alignas(1024) uint8_t ring[2][2 * kHalfBytes];
  alignas(1024) uint8_t ds[2 * kHalfBytes];
  alignas(16) float lse2[2][128];
  alignas(16) float dvec_s[2][128];
  uint64_t kv_full;
  uint64_t q_full[2];   // LSE / D rows of an item (32 producer lanes)
  uint64_t q_empty[2];
  uint64_t r_full[2], r_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, dq_free, done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdSmem<256>) <= 232448, "head dim 256: shared memory");

struct BwdKernelArgs {
  BwdArgs a;
};

__device__ __forceinline__ int block_of(const int32_t* offs, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Iterates the (query head in group, list index) pairs of one CTA in order,
// for the group's query heads [h_lo, h_hi).  Chunked units (kChunked) take
// only the entries whose query tile lies in [qlo, qhi): each list is sorted
// by query tile, so that is a contiguous index range, found by two binary
// searches per head.
template <bool kChunked>
struct ItemIter {
  const int32_t* cnt_base;  // bwd_cnt for (b, list head 0), stride nKt per list head
  const int32_t* lst_base;
  int nH, nKt, nQt, kt, G, g, hend, qlo, qhi;
  int hi, idx, cnt, cur;
  __device__ void init(const TileMetaDev& t, int b, int kt_, int G_, int g_, int h_lo, int h_hi,
                       int qlo_ = 0, int qhi_ = 0) {
    nH = t.nH; nKt = t.nKt; nQt = t.nQt; kt = kt_; G = G_; g = g_; hend = h_hi; qlo = qlo_; qhi = qhi_;
    cnt_base = t.bwd_cnt + (int64_t)b * t.nH * t.nKt;
    lst_base = t.bwd_lst + (int64_t)b * t.nH * t.nKt * t.nQt;
    hi = h_lo; idx = 0;
    cnt = 0;
    if (hi < hend) range_of(hi);
    skip_empty();
  }
  __device__ int list_head(int hh) const { return nH == 1 ? 0 : g * G + hh; }
  __device__ int count_of(int hh) const { return __ldg(cnt_base + (int64_t)list_head(hh) * nKt + kt); }
  // First index in [0, n) of list `l` whose query tile is >= q (n if none).
  __device__ int lower(const int32_t* l, int n, int q) const {
    int lo = 0, hi_ = n;
    while (lo < hi_) {
      const int mid = (lo + hi_) >> 1;
      if ((__ldg(l + mid) >> 1) < q) lo = mid + 1; else hi_ = mid;
    }
    return lo;
  }
  __device__ void range_of(int hh) {
    cnt = count_of(hh);
    idx = 0;
    if (kChunked) {
      const int32_t* l = lst_base + ((int64_t)list_head(hh) * nKt + kt) * nQt;
      idx = lower(l, cnt, qlo);
      cnt = lower(l, cnt, qhi);
    }
  }
  // Advances past empty lists and loads the entry at the new position early,
  // so the load overlaps the rest of the current iteration.
  __device__ void skip_empty() {
    while (hi < hend && idx >= cnt) { ++hi; if (hi < hend) range_of(hi); }
    if (hi < hend) cur = __ldg(lst_base + ((int64_t)list_head(hi) * nKt + kt) * nQt + idx);
  }
  __device__ bool valid() const { return hi < hend; }
  __device__ int entry() const { return cur; }
  __device__ int head() const { return g * G + hi; }
  __device__ void next() { ++idx; skip_empty(); }
};

// Bits [lo, hi) of a 64-bit column mask that fall into the word starting at `base`.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int base) {
  const int a = max(lo, base), b = min(hi, base + 32);
  if (b <= a) return 0u;
  const int n = b - a;
  return (n == 32) ? 0xffffffffu : (((1u << n) - 1u) << (a - base));
}

// kDq = false: the dQ product, its drain and the dS^T copy in shared memory
// are left out (dQ then comes from the separate dQ kernel, dq.cu).
template <int D, bool kChunked, bool kDq>
__global__ void __launch_bounds__(kThreadsDkdv, 1)
dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
            const __grid_constant__ BwdKernelArgs ka) {
  constexpr int kTileBytes = BwdGeom<D>::kTileBytes;
  constexpr int kBoxes = BwdGeom<D>::kBoxes;
  static_assert(D != 256 || kDq, "head dim 256 has no separate dQ kernel");
  constexpr int kOut = D == 256 ? 128 : D;  // head-dim columns of dK / dV / dQ this unit owns
  // TMEM columns of dK and dQ^T (dQ^T has a region of its own at D = 64).
  constexpr bool kSepDq = D == 64;
  constexpr uint32_t kColDK = D == 64 ? 320 : 384;
  constexpr uint32_t kColDQ = kSepDq ? 384 : 128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const BwdArgs& a = ka.a;
  const ProblemDev& pr = a.pr;
  int32_t* gstatus = a.meta.status;
  if ((smem_u32(smem_raw) & 1023u) != 0u) {  // layout relies on 1 KB alignment
    if (threadIdx.x == 0) atomicCAS(gstatus, 0, LCATTN_ERR_CUDA);
    return;
  }
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Chunked units (per-head lists): blockIdx.z = batch * nchunks + query chunk,
  // so the units launched one after another share a chunk of query tiles.
  const int b = kChunked ? (int)(blockIdx.z / a.nchunks) : (int)blockIdx.z;
  const int chunk = kChunked ? (int)(blockIdx.z % a.nchunks) : 0;
  const int qlo = chunk * a.chunk_tiles, qhi = min(a.meta.nQt, qlo + a.chunk_tiles);
  const int g = blockIdx.y;
  // Longest key tiles first.  With per-head lists the order of the group's
  // first head is used.  With a split, the parts of one key tile (shares of
  // the group's query heads) are adjacent CTAs; at D = 256 the two head-dim
  // halves of a unit are adjacent too.
  const int hd = D == 256 ? (int)(blockIdx.x & 1u) : 0;
  const int col0 = hd * 128;  // first head-dim column this unit owns
  const int ux = D == 256 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int parts = a.parts;
  const int part = ux % parts;
  const int h_lo = part * pr.G / parts, h_hi = (part + 1) * pr.G / parts;
  const int lh0 = a.meta.nH == 1 ? 0 : g * pr.G;
  const int kt = __ldg(a.meta.bwd_ord + ((int64_t)b * a.meta.nH + lh0) * a.meta.nKt + ux / parts);

  if (tid == 0) {
    mbar_init(&sm.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], D == 256 ? 32 : 33);  // (+ the expect-tx arrival of the Q/dO tiles)
      mbar_init(&sm.q_empty[s], 1);
    }
    if constexpr (D == 256) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(&sm.r_full[s], 1);
        mbar_init(&sm.r_empty[s], 1);
      }
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.p_ready, 256);
    mbar_init(&sm.ds_ready, 256);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, 128);
    mbar_init(&sm.done, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) tmem_alloc(&sm.tmem_base, 512);
  if (D == 64) {
    // Zero half of the K buffer: head-dim rows 64-127 of the padded dQ^T
    // product.  Written by the generic proxy, read by the tensor cores.
    reinterpret_cast<uint4*>(sm.k + kHalfBytes)[tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(sm.k + kHalfBytes)[tid + kThreadsDkdv] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  const int TO = LCATTN_ERR_DEVICE_TIMEOUT;

  if (warp >= 12) {
    regs_dec<BwdRegs<D, kDq>::kCtl>();
  if (warp == 12) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; the elected lane issues the copies.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    mbar_expect_tx_e(&sm.kv_full, 2 * kTileBytes);
    for (int bx = 0; bx < kBoxes; ++bx) {
      tma_load_4d_e(sm.k + bx * kHalfBytes, &tmK, &sm.kv_full, 64 * bx, g, kt * kBN, b);
      tma_load_4d_e(sm.v + bx * kHalfBytes, &tmV, &sm.kv_full, 64 * bx, g, kt * kBN, b);
    }
    ItemIter<kChunked> it;
    it.init(a.meta, b, kt, pr.G, g, h_lo, h_hi, qlo, qhi);
    // LSE / D rows of item i (query tile qt of head h) into row slot i & 1, stored
    // negated: -(LSE*log2(e) - log2(scale)) (-inf for a fully masked row: P = 0) and -D.
    auto stage_rows = [&](int st, int h, int qt) {
      const float log2_scale = log2f(a.scale);
      const float* lse = a.lse + ((int64_t)b * pr.Hq + h) * pr.Sq;
      const float* dv = a.dvec + ((int64_t)b * pr.Hq + h) * pr.Sq;
      #pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = lane * 4 + k;
        const int q = qt * kBM + c;
        float l2 = -INFINITY, d = 0.f;
        if (q < pr.Sq) {
          const float l = __ldg(lse + q);
          l2 = (l == -INFINITY) ? -INFINITY : log2_scale - l * kLog2e;
          d = __ldg(dv + q);
        }
        sm.lse2[st][c] = l2;
        sm.dvec_s[st][c] = -d;
      }
    };
    if constexpr (D == 256) {
      // Ring entries in the MMA warp's order: Q(0) and dO(0) (both halves),
      // then per item i: the own half of dO(i) (dV), Q(i+1) (S^T), the own half
      // of Q(i) (dK), dO(i+1) (dP^T).
      int t = 0;  // ring entries issued
      auto load_half = [&](const CUtensorMap* tm, int h, int qt, int half) -> bool {
        const int stg = t & 1, use = t >> 1;
        if (use > 0) {
          const bool w = mbar_wait(&sm.r_empty[stg], (use - 1) & 1, abort_flag, gstatus, TO);
          if (!__all_sync(0xffffffffu, w)) return false;
        }
        mbar_expect_tx_e(&sm.r_full[stg], 2 * kHalfBytes);
        tma_load_4d_e(sm.ring[stg], tm, &sm.r_full[stg], 128 * half, h, qt * kBM, b);
        tma_load_4d_e(sm.ring[stg] + kHalfBytes, tm, &sm.r_full[stg], 128 * half + 64, h, qt * kBM, b);
        ++t;
        return true;
      };
      auto load_rows = [&](int i, int h, int qt) -> bool {
        const int st = i & 1, use = i >> 1;
        if (use > 0) {
          const bool w = mbar_wait(&sm.q_empty[st], (use - 1) & 1, abort_flag, gstatus, TO);
          if (!__all_sync(0xffffffffu, w)) return false;
        }
        stage_rows(st, h, qt);
        mbar_arrive(&sm.q_full[st]);
        return true;
      };
      if (it.valid()) {
        int h = it.head(), qt = it.entry() >> 1;
        bool ok = load_rows(0, h, qt) && load_half(&tmQ, h, qt, 0) && load_half(&tmQ, h, qt, 1) &&
                  load_half(&tmdO, h, qt, 0) && load_half(&tmdO, h, qt, 1);
        for (int i = 0; ok; ++i) {
          it.next();
          const bool more = it.valid();
          const int h2 = more ? it.head() : 0, qt2 = more ? it.entry() >> 1 : 0;
          ok = load_half(&tmdO, h, qt, hd);
          if (ok && more) ok = load_rows(i + 1, h2, qt2) && load_half(&tmQ, h2, qt2, 0) && load_half(&tmQ, h2, qt2, 1);
          if (ok) ok = load_half(&tmQ, h, qt, hd);
          if (ok && more) ok = load_half(&tmdO, h2, qt2, 0) && load_half(&tmdO, h2, qt2, 1);
          if (!more) break;
          h = h2;
          qt = qt2;
        }
      }
      // Never leave copies in flight (bounded waits that ignore the abort word).
      int dummy = 0;
      for (int u = max(0, t - 2); u < t; ++u) mbar_wait(&sm.r_full[u & 1], (u >> 1) & 1, &dummy, gstatus, TO);
      mbar_wait(&sm.kv_full, 0, &dummy, gstatus, TO);
    } else {
    int i = 0, issued = 0;
    for (; it.valid(); it.next(), ++i) {
      const int st = i & 1, use = i >> 1;
      if (use > 0) {
        bool ok = mbar_wait(&sm.q_empty[st], (use - 1) & 1, abort_flag, gstatus, TO);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int qt = it.entry() >> 1;
      const int h = it.head();
      mbar_expect_tx_e(&sm.q_full[st], 2 * kTileBytes);
      for (int bx = 0; bx < kBoxes; ++bx) {
        tma_load_4d_e(sm.q[st] + bx * kHalfBytes, &tmQ, &sm.q_full[st], 64 * bx, h, qt * kBM, b);
        tma_load_4d_e(sm.dO[st] + bx * kHalfBytes, &tmdO, &sm.q_full[st], 64 * bx, h, qt * kBM, b);
      }
      stage_rows(st, h, qt);
      mbar_arrive(&sm.q_full[st]);
      issued = i + 1;
    }
    {
      int dummy = 0;
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait(&sm.q_full[t & 1], (t >> 1) & 1, &dummy, gstatus, TO);
      mbar_wait(&sm.kv_full, 0, &dummy, gstatus, TO);
    }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    // Per item i: wait P'(i) | dV(i) | S^T(i+1) | wait dS(i) | dK(i) | dQ^T(i) |
    // wait drain | dP^T(i+1).  dV needs only P', so S^T(i+1) can follow it
    // while dS(i) is still being formed, and P'(i+1) starts right after.  The
    // whole warp runs the loop; each tcgen05.mma / commit is issued by one
    // elected lane.
    if constexpr (D == 256) {
      // Head dim 256: the same order, with S^T / dP^T over both halves of the
      // head dim (two ring entries each) and dV / dK / dQ^T over the own half.
      const uint32_t id_kmaj = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_ts = idesc_bf16_f32(128, 128, false, true);
      const uint32_t id_mn = idesc_bf16_f32(128, 128, true, true);
      const uint32_t tS = tmem, tP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
      const uint64_t dK_k = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t dV_k = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(smem_u32(sm.k + hd * 2 * kHalfBytes), kHalfBytes, 1024);
      const uint64_t r_k = sdesc_sw128(smem_u32(sm.ring[0]), 16, 1024);
      const uint64_t r_mn = sdesc_sw128(smem_u32(sm.ring[0]), kHalfBytes, 1024);
      const uint64_t dS_mn = sdesc_sw128(smem_u32(sm.ds), kHalfBytes, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.kv_full, 0, abort_flag, gstatus, TO));
      ItemIter<kChunked> it;
      it.init(a.meta, b, kt, pr.G, g, h_lo, h_hi, qlo, qhi);
      int t = 0;  // ring entries consumed
      // Waits for ring entry t; its stage, or -1 when the wait gave up.
      auto take = [&]() -> int {
        const int stg = t & 1;
        const bool w = mbar_wait(&sm.r_full[stg], (t >> 1) & 1, abort_flag, gstatus, TO);
        if (!__all_sync(0xffffffffu, w)) return -1;
        tc_fence_after();
        return stg;
      };
      // d = A B^T over the whole head dim: A = K or V (resident, K-major), B =
      // the two halves of a Q or dO tile (ring entries, K-major).
      auto full_prod = [&](uint32_t d, uint64_t a_base) -> bool {
        for (int half = 0; half < 2; ++half) {
          const int stg = take();
          if (stg < 0) return false;
          const uint64_t a0 = sdesc_add(a_base, half * 2 * kHalfBytes);
          const uint64_t b0 = sdesc_add(r_k, stg * 2 * kHalfBytes);
          if (half == 0) mma_ss_e<0>(d, a0, b0, id_kmaj);
          else mma_ss_e<1>(d, a0, b0, id_kmaj);
          #pragma unroll
          for (int kk = 1; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            mma_ss_e<1>(d, sdesc_add(a0, off), sdesc_add(b0, off), id_kmaj);
          }
          tc_commit_e(&sm.r_empty[stg]);
          ++t;
        }
        return true;
      };
      // d (+)= A B: A = P'^T or dS^T from TMEM, B = the own half of dO or Q (MN-major).
      auto half_prod = [&](uint32_t d, uint32_t a_tm, uint32_t acc) -> bool {
        const int stg = take();
        if (stg < 0) return false;
        const uint64_t b0 = sdesc_add(r_mn, stg * 2 * kHalfBytes);
        mma_ts_er(d, a_tm, b0, id_ts, acc);
        #pragma unroll
        for (int kk = 1; kk < 8; ++kk)
          mma_ts_e<1>(d, a_tm + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_add(b0, kk * 2048), id_ts);
        tc_commit_e(&sm.r_empty[stg]);
        ++t;
        return true;
      };
      if (ok && it.valid()) {
        ok = full_prod(tS, dK_k);  // S^T(0)
        if (ok) tc_commit_e(&sm.s_full);
        if (ok) ok = full_prod(tP, dV_k);  // dP^T(0)
        if (ok) tc_commit_e(&sm.dp_full);
      }
      for (int i = 0; ok && it.valid(); ++i) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_ready, i & 1, abort_flag, gstatus, TO));
        if (!ok) break;
        tc_fence_after();
        if (!(ok = half_prod(tdV, tS, i > 0 ? 1u : 0u))) break;  // dV(i)
        it.next();
        const bool more = it.valid();
        if (more) {
          if (!(ok = full_prod(tS, dK_k))) break;  // S^T(i+1)
          tc_commit_e(&sm.s_full);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.ds_ready, i & 1, abort_flag, gstatus, TO));
        if (!ok) break;
        tc_fence_after();
        if (!(ok = half_prod(tdK, tP, i > 0 ? 1u : 0u))) break;  // dK(i)
        tc_commit_e(&sm.q_empty[i & 1]);  // LSE(i), D(i) are read for good
        // dQ^T (own half) = K_half^T dS^T into [128, 256).
        mma_ss_e<0>(tP, dK_mn, dS_mn, id_mn);
        #pragma unroll
        for (int kk = 1; kk < 8; ++kk)
          mma_ss_e<1>(tP, sdesc_add(dK_mn, kk * 2048), sdesc_add(dS_mn, kk * 2048), id_mn);
        tc_commit_e(&sm.dq_full);
        if (more) {
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.dq_free, i & 1, abort_flag, gstatus, TO));
          if (!ok) break;
          tc_fence_after();
          if (!(ok = full_prod(tP, dV_k))) break;  // dP^T(i+1)
          tc_commit_e(&sm.dp_full);
        }
      }
      tc_commit_e(&sm.done);
      int dummy = 0;
      mbar_wait(&sm.done, 0, &dummy, gstatus, TO);
    } else
    {
      const uint32_t id_kmaj = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_ts = idesc_bf16_f32(128, D, false, true);
      const uint32_t id_mn = idesc_bf16_f32(128, 128, true, true);
      const uint32_t tS = tmem, tP = tmem + 128, tdV = tmem + 256, tdK = tmem + kColDK;
      const uint32_t tQd = tmem + kColDQ;
      // Base descriptors (K-major and MN-major views); ring stage st is kTileBytes on.
      const uint64_t dK_k = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(smem_u32(sm.k), kHalfBytes, 1024);
      const uint64_t dV_k = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      const uint64_t dQ_k = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dQ_mn = sdesc_sw128(smem_u32(sm.q[0]), kHalfBytes, 1024);
      const uint64_t dO_k = sdesc_sw128(smem_u32(sm.dO[0]), 16, 1024);
      const uint64_t dO_mn = sdesc_sw128(smem_u32(sm.dO[0]), kHalfBytes, 1024);
      const uint64_t dS_mn = sdesc_sw128(smem_u32(sm.ds), kHalfBytes, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.kv_full, 0, abort_flag, gstatus, TO));
      ItemIter<kChunked> it;
      it.init(a.meta, b, kt, pr.G, g, h_lo, h_hi, qlo, qhi);
      // Both operands K-major: 16-column steps inside a 64-column half, then the next half.
      auto issue_kmaj = [&](uint32_t d, uint64_t a0, uint64_t b0) {
        mma_ss_e<0>(d, a0, b0, id_kmaj);
        #pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_ss_e<1>(d, sdesc_add(a0, off), sdesc_add(b0, off), id_kmaj);
        }
      };
      // Prologue: S^T(0) and dP^T(0).
      if (ok && it.valid()) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full[0], 0, abort_flag, gstatus, TO));
        if (ok) {
          tc_fence_after();
          issue_kmaj(tS, dK_k, dQ_k);  // S^T(0) = K Q_0^T
          tc_commit_e(&sm.s_full);
          issue_kmaj(tP, dV_k, dO_k);  // dP^T(0) = V dO_0^T
          tc_commit_e(&sm.dp_full);
        }
      }
      int i = 0;
      for (; ok && it.valid(); ++i) {
        const int st = i & 1;
        const uint32_t qoff = st * kTileBytes;
        // dV += P'^T dO as soon as P'(i) is in TMEM (A from TMEM: queries 0-63
        // sit in the first 32 columns of each half's region, 64-127 at +64).
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_ready, i & 1, abort_flag, gstatus, TO));
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t bo = sdesc_add(dO_mn, qoff);
          mma_ts_er(tdV, tS, bo, id_ts, i > 0 ? 1u : 0u);
          #pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ts_e<1>(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_add(bo, kk * 2048), id_ts);
        }
        // S^T(i+1) right behind it: it overwrites P'(i), which dV(i) read
        // before (in-order), and the elementwise pass keeps P' in registers.
        it.next();
        const bool more = it.valid();
        if (more) {
          const int st2 = (i + 1) & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full[st2], ((i + 1) >> 1) & 1, abort_flag, gstatus, TO));
          if (!ok) break;
          tc_fence_after();
          issue_kmaj(tS, dK_k, sdesc_add(dQ_k, st2 * kTileBytes));  // S^T(i+1)
          tc_commit_e(&sm.s_full);
        }
        // dK += dS^T Q once dS(i) is ready (A = dS^T from TMEM).
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.ds_ready, i & 1, abort_flag, gstatus, TO));
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t bq = sdesc_add(dQ_mn, qoff);
          mma_ts_er(tdK, tP, bq, id_ts, i > 0 ? 1u : 0u);
          #pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ts_e<1>(tdK, tP + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_add(bq, kk * 2048), id_ts);
        }
        tc_commit_e(&sm.q_empty[st]);  // Q(i), dO(i), LSE(i), D(i) are read for good
        if (kDq) {
          // dQ^T = K^T dS^T: A = K read MN-major (M = head dim), B = dS^T read
          // MN-major (N = queries).  Lands in [128, 256) (D = 64: [384, 512),
          // once the drain has read dQ^T(i-1) there): lane = head dim.
          if (kSepDq && i > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.dq_free, (i - 1) & 1, abort_flag, gstatus, TO));
            if (!ok) break;
            tc_fence_after();
          }
          mma_ss_e<0>(tQd, dK_mn, dS_mn, id_mn);
          #pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ss_e<1>(tQd, sdesc_add(dK_mn, kk * 2048), sdesc_add(dS_mn, kk * 2048), id_mn);
          tc_commit_e(&sm.dq_full);
        }
        // dP^T(i+1) = V dO^T, into the columns dQ^T(i) uses: wait for its drain
        // (without the dQ product, dK(i) read dS^T(i) from them first, in order;
        // at D = 64 dQ^T has columns of its own).
        if (more) {
          if (kDq && !kSepDq) {
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.dq_free, i & 1, abort_flag, gstatus, TO));
            if (!ok) break;
          }
          tc_fence_after();
          issue_kmaj(tP, dV_k, sdesc_add(dO_k, ((i + 1) & 1) * kTileBytes));
          tc_commit_e(&sm.dp_full);
        }
      }
      tc_commit_e(&sm.done);
      int dummy = 0;
      mbar_wait(&sm.done, 0, &dummy, gstatus, TO);
    }
  }
  } else if (warp >= 8) {
    regs_inc<BwdRegs<D, kDq>::kDrain>();
    // ------------------------------------------------------------ dQ drain
    if (kDq) {
    const int r = 32 * (warp & 3) + lane;  // head-dim row of dQ^T (TMEM lane)
    const uint32_t tQ = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kColDQ;
    const int64_t dq_row_stride = a.dqa_ss;
    ItemIter<kChunked> it;
    it.init(a.meta, b, kt, pr.G, g, h_lo, h_hi, qlo, qhi);
    for (int i = 0; it.valid(); it.next(), ++i) {
      const int qt = it.entry() >> 1;
      const int h = it.head();
      bool ok = mbar_wait(&sm.dq_full, i & 1, abort_flag, gstatus, TO);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (r >= D) {  // zero rows of the padded product (D = 64): nothing to add
        mbar_arrive(&sm.dq_free);
        continue;
      }
      tc_fence_after();
      uint32_t d[128];
      tmem_ld32(tQ, d);
      tmem_ld32(tQ + 32, d + 32);
      tmem_ld32(tQ + 64, d + 64);
      tmem_ld32(tQ + 96, d + 96);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.dq_free);  // columns [128, 256) may take dP^T(i+1) now
      const int q0 = qt * kBM;
      const int nq = min(kBM, pr.Sq - q0);
      float* dst = a.dq_acc + (int64_t)b * a.dqa_sb + (int64_t)q0 * a.dqa_ss + (int64_t)h * a.dqa_sh + col0 + r;
      if (nq == kBM) {
        #pragma unroll
        for (int c = 0; c < 128; ++c) atomicAdd(dst + c * dq_row_stride, __uint_as_float(d[c]));
      } else {
        #pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < nq) atomicAdd(dst + c * dq_row_stride, __uint_as_float(d[c]));
      }
    }
    }
  } else {
    regs_inc<kRegsWork>();
    // ------------------------------------------------------------ elementwise
    // Warpgroup x takes query columns [64x, 64x+64) of every tile; thread r is
    // key row r of S^T / dP^T (the TMEM lane).
    const int x = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int c0 = 64 * x;
    const int key = kt * kBN + r;
    const bool key_ok = key < pr.Sk;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_off, tP = tmem + lane_off + 128;
    const float sl2 = a.scale_log2;
    int4 cb = make_int4(0, 0, 0, 0);
    int kb = 0;
    if (key_ok) {
      if (a.mask.kind == LCATTN_MASK_COLBOUNDS) cb = __ldg(a.mask.col_bounds + (int64_t)b * pr.Sk + key);
      else kb = block_of(a.mask.k_offs, a.mask.nKb, key);
    }
    ItemIter<kChunked> it;
    it.init(a.meta, b, kt, pr.G, g, h_lo, h_hi, qlo, qhi);
    int i = 0;
    bool ok = true;
    for (; it.valid(); it.next(), ++i) {
      const int st = i & 1;
      const int e = it.entry();
      const int qt = e >> 1;
      const int h = it.head();
      const int q0 = qt * kBM + c0;
      // Per-element mask only for partial tiles and keys past Sk (warp-uniform
      // except for the key test, which is per lane).
      const bool masked = (e & 1) != 0 || !key_ok;
      uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
      if (!key_ok) {
        m0 = m1 = 0u;
      } else if (masked) {
        if (a.mask.kind == LCATTN_MASK_COLBOUNDS) {
          // This key's allowed query rows [a0, b0) U [a1, b1), clipped to the
          // 64 columns [q0, q0 + 64) of this warpgroup: two bit ranges.
          const int lo0 = max(cb.x, q0) - q0, hi0 = min(cb.y, q0 + 64) - q0;
          const int lo1 = max(cb.z, q0) - q0, hi1 = min(cb.w, q0 + 64) - q0;
          m0 = range_bits(lo0, hi0, 0) | range_bits(lo1, hi1, 0);
          m1 = range_bits(lo0, hi0, 32) | range_bits(lo1, hi1, 32);
        } else {
          m0 = m1 = 0u;
          const uint8_t* map = a.mask.block_map +
                               ((int64_t)b * pr.Hq + h) * a.mask.nQb * (int64_t)a.mask.nKb + kb;
          const int q1 = min(q0 + 64, pr.Sq);
          for (int qb = block_of(a.mask.q_offs, a.mask.nQb, min(q0, pr.Sq - 1)); qb < a.mask.nQb; ++qb) {
            const int lo = max(__ldg(a.mask.q_offs + qb), q0);
            if (lo >= q1) break;
            const int hi = min(__ldg(a.mask.q_offs + qb + 1), q1);
            if (hi > lo && __ldg(map + (int64_t)qb * a.mask.nKb)) {
              m0 |= range_bits(lo - q0, hi - q0, 0);
              m1 |= range_bits(lo - q0, hi - q0, 32);
            }
          }
        }
      }
      // Rows past Sq carry a negated LSE of -inf (set by the producer), so P = 0 there.
      ok = mbar_wait(&sm.q_full[st], (i >> 1) & 1, abort_flag, gstatus, TO) &&
           mbar_wait(&sm.s_full, i & 1, abort_flag, gstatus, TO);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const float4* lse4 = reinterpret_cast<const float4*>(sm.lse2[st] + c0);
      const float4* dv4 = reinterpret_cast<const float4*>(sm.dvec_s[st] + c0);
      // ---- P'^T = scale * P^T for 64 queries, bf16 into TMEM (kept packed)
      uint32_t pk[32];
      {
        uint32_t s0[32], s1[32];
        tmem_ld32(tS + c0, s0);
        tmem_ld32(tS + c0 + 32, s1);
        tmem_ld_wait();
        const float2 sl2v = make_float2(sl2, sl2);
        #pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 la = lse4[c4], lb = lse4[8 + c4];
          // exp2(S * scale * log2(e) + (-lse2)) on column pairs (paired fp32 FMA).
          const float2 ya0 = fma2(make_float2(__uint_as_float(s0[4 * c4]), __uint_as_float(s0[4 * c4 + 1])),
                                  sl2v, make_float2(la.x, la.y));
          const float2 ya1 = fma2(make_float2(__uint_as_float(s0[4 * c4 + 2]), __uint_as_float(s0[4 * c4 + 3])),
                                  sl2v, make_float2(la.z, la.w));
          const float2 yb0 = fma2(make_float2(__uint_as_float(s1[4 * c4]), __uint_as_float(s1[4 * c4 + 1])),
                                  sl2v, make_float2(lb.x, lb.y));
          const float2 yb1 = fma2(make_float2(__uint_as_float(s1[4 * c4 + 2]), __uint_as_float(s1[4 * c4 + 3])),
                                  sl2v, make_float2(lb.z, lb.w));
          float pa[4] = {fast_exp2(ya0.x), fast_exp2(ya0.y), fast_exp2(ya1.x), fast_exp2(ya1.y)};
          float pb[4] = {fast_exp2(yb0.x), fast_exp2(yb0.y), fast_exp2(yb1.x), fast_exp2(yb1.y)};
          if (masked) {
            #pragma unroll
            for (int u = 0; u < 4; ++u) {
              pa[u] = ((m0 >> (4 * c4 + u)) & 1u) ? pa[u] : 0.f;
              pb[u] = ((m1 >> (4 * c4 + u)) & 1u) ? pb[u] : 0.f;
            }
          }
          pk[2 * c4] = pack_bf16x2(pa[0], pa[1]);
          pk[2 * c4 + 1] = pack_bf16x2(pa[2], pa[3]);
          pk[16 + 2 * c4] = pack_bf16x2(pb[0], pb[1]);
          pk[16 + 2 * c4 + 1] = pack_bf16x2(pb[2], pb[3]);
        }
        tmem_st32(tS + c0, pk);  // columns [64x, 64x + 32): only this warpgroup read them
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_ready);  // dV(i) may start; P' stays in registers for dS
      }
      // ---- dS^T = P'^T (dP^T - D) = scale * P^T (dP^T - D), from the bf16 P'
      ok = mbar_wait(&sm.dp_full, i & 1, abort_flag, gstatus, TO);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t d0[32], d1[32];
        tmem_ld32(tP + c0, d0);
        tmem_ld32(tP + c0 + 32, d1);
        tmem_ld_wait();
        uint32_t dk[32];
        #pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 da = dv4[c4], db = dv4[8 + c4];
          // dP - D on column pairs (fp32), rounded to bf16 pairs, times the bf16
          // P' pairs on the packed bf16 ALU: dS^T leaves in bf16 either way.
          const float2 ta0 = add2(make_float2(__uint_as_float(d0[4 * c4]), __uint_as_float(d0[4 * c4 + 1])),
                                  make_float2(da.x, da.y));
          const float2 ta1 = add2(make_float2(__uint_as_float(d0[4 * c4 + 2]), __uint_as_float(d0[4 * c4 + 3])),
                                  make_float2(da.z, da.w));
          const float2 tb0 = add2(make_float2(__uint_as_float(d1[4 * c4]), __uint_as_float(d1[4 * c4 + 1])),
                                  make_float2(db.x, db.y));
          const float2 tb1 = add2(make_float2(__uint_as_float(d1[4 * c4 + 2]), __uint_as_float(d1[4 * c4 + 3])),
                                  make_float2(db.z, db.w));
          dk[2 * c4] = mul_bf16x2(pk[2 * c4], pack_bf16x2(ta0.x, ta0.y));
          dk[2 * c4 + 1] = mul_bf16x2(pk[2 * c4 + 1], pack_bf16x2(ta1.x, ta1.y));
          dk[16 + 2 * c4] = mul_bf16x2(pk[16 + 2 * c4], pack_bf16x2(tb0.x, tb0.y));
          dk[16 + 2 * c4 + 1] = mul_bf16x2(pk[16 + 2 * c4 + 1], pack_bf16x2(tb1.x, tb1.y));
        }
        tmem_st32(tP + c0, dk);
        if (kDq) {
          // dS^T row r, queries [64x, 64x+64) -> 8 swizzled 16-byte chunks of half x.
          uint8_t* ds_row = sm.ds + x * kHalfBytes + r * 128;
          #pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(ds_row + ((u ^ (r & 7)) << 4)) =
                make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tmem_st_wait();
      if (kDq) fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.ds_ready);
    }
    // ---- dV (warpgroup 0) / dK (warpgroup 1) out, bf16; zero when no query
    // tile touched this key tile.  dV accumulated P' = scale * P: undo it.
    // In accumulate mode the fp32 values are reduce-added into the caller's
    // accumulators instead (nothing to add when no query tile touched the tile).
    const bool red_out = a.accum || kChunked;
    if (ok && !(red_out && i == 0)) {
      bool have = i > 0;
      if (have) {
        have = mbar_wait(&sm.done, 0, abort_flag, gstatus, TO);
        have = __all_sync(0xffffffffu, have);
        tc_fence_after();
      }
      const float mul = x == 0 ? 1.f / a.scale : 1.f;
      const uint32_t tacc = tmem + lane_off + (x == 0 ? 256 : kColDK);
      // Split units write fp32 partials [part][dV, dK][B][Sk][Hkv][D]; a
      // reduction kernel sums the parts into the bf16 outputs.
      float* pdst = a.dkv_part + (((((int64_t)part * 2 + x) * pr.B + b) * pr.Sk + key) * pr.Hkv + g) * D + col0;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(x == 0 ? a.dv : a.dk) +
                           (int64_t)b * (x == 0 ? a.v_sb : a.k_sb) +
                           (int64_t)key * (x == 0 ? a.v_ss : a.k_ss) +
                           (int64_t)g * (x == 0 ? a.v_sh : a.k_sh);
      #pragma unroll
      for (int c = 0; c < kOut / 32; ++c) {
        uint32_t xr[32];
        if (have) {
          tmem_ld32(tacc + c * 32, xr);
          tmem_ld_wait();
        } else {
          #pragma unroll
          for (int k = 0; k < 32; ++k) xr[k] = 0u;
        }
        if (key_ok && red_out) {
          float* adst = (x == 0 ? a.dv_acc : a.dk_acc) + (((int64_t)b * pr.Sk + key) * pr.Hkv + g) * D + col0 + c * 32;
          #pragma unroll
          for (int u = 0; u < 8; ++u)
            red_add_v4(adst + 4 * u, __uint_as_float(xr[4 * u]) * mul, __uint_as_float(xr[4 * u + 1]) * mul,
                       __uint_as_float(xr[4 * u + 2]) * mul, __uint_as_float(xr[4 * u + 3]) * mul);
        } else if (key_ok && parts > 1) {
          float4* p4 = reinterpret_cast<float4*>(pdst + c * 32);
          #pragma unroll
          for (int u = 0; u < 8; ++u)
            p4[u] = make_float4(__uint_as_float(xr[4 * u]) * mul, __uint_as_float(xr[4 * u + 1]) * mul,
                                __uint_as_float(xr[4 * u + 2]) * mul, __uint_as_float(xr[4 * u + 3]) * mul);
        } else if (key_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + col0 + c * 32);
          #pragma unroll
          for (int u = 0; u < 4; ++u)
            d4[u] = make_uint4(
                pack_bf16x2(__uint_as_float(xr[8 * u]) * mul, __uint_as_float(xr[8 * u + 1]) * mul),
                pack_bf16x2(__uint_as_float(xr[8 * u + 2]) * mul, __uint_as_float(xr[8 * u + 3]) * mul),
                pack_bf16x2(__uint_as_float(xr[8 * u + 4]) * mul, __uint_as_float(xr[8 * u + 5]) * mul),
                pack_bf16x2(__uint_as_float(xr[8 * u + 6]) * mul, __uint_as_float(xr[8 * u + 7]) * mul));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 13) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kChunked, bool kDq>
cudaError_t launch_dkdv_dc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
  static bool attr_done = false;
  const size_t smem = sizeof(BwdSmem<D>);
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(dkdv_kernel<D, kChunked, kDq>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  BwdKernelArgs ka;
  ka.a = a;
  dim3 grid(a.meta.nKt * a.parts * (D == 256 ? 2 : 1), a.pr.Hkv, a.pr.B * a.nchunks);
  dkdv_kernel<D, kChunked, kDq><<<grid, kThreadsDkdv, smem, st>>>(tq, tk, tv, tdo, ka);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dkdv_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
  cudaError_t e;
  if constexpr (D == 256) {
    if (a.dq_sep) return cudaErrorInvalidValue;  // no dQ kernel at D = 256
    e = a.nchunks > 1 ? launch_dkdv_dc<D, true, true>(tq, tk, tv, tdo, a, st)
                      : launch_dkdv_dc<D, false, true>(tq, tk, tv, tdo, a, st);
  } else if (a.dq_sep)
    e = a.nchunks > 1 ? launch_dkdv_dc<D, true, false>(tq, tk, tv, tdo, a, st)
                      : launch_dkdv_dc<D, false, false>(tq, tk, tv, tdo, a, st);
  else
    e = a.nchunks > 1 ? launch_dkdv_dc<D, true, true>(tq, tk, tv, tdo, a, st)
                      : launch_dkdv_dc<D, false, true>(tq, tk, tv, tdo, a, st);
  // Split or chunked units leave fp32 dK/dV (partials, or one accumulator):
  // sum / convert them into the bf16 outputs.  The accumulate mode keeps fp32.
  if (e != cudaSuccess || a.accum || a.red_parts == 0) return e;
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n = 2 * (int64_t)a.pr.B * a.pr.Sk * a.pr.Hkv * (D / 8);
  int64_t blocks = (n + 255) / 256;
  if (blocks > (int64_t)nsm * 16) blocks = (int64_t)nsm * 16;
  dkv_reduce_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prepass(const BwdArgs& a, cudaStream_t st) {
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > (int64_t)nsm * 32) blocks = (int64_t)nsm * 32;
  if (a.pr.D == 64) prepass_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(a);
  else if (a.pr.D == 256) prepass_kernel<256><<<(unsigned)blocks, 256, 0, st>>>(a);
  else prepass_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
  if (a.pr.D == 64) return launch_dkdv_d<64>(tq, tk, tv, tdo, a, st);
  if (a.pr.D == 256) return launch_dkdv_d<256>(tq, tk, tv, tdo, a, st);
  return launch_dkdv_d<128>(tq, tk, tv, tdo, a, st);
}

cudaError_t launch_bwd_dq_convert(const BwdArgs& a, cudaStream_t st) {
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nvec = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq * (a.pr.D / 8);
  int64_t blocks = (nvec + 255) / 256;
  if (blocks > (int64_t)nsm * 32) blocks = (int64_t)nsm * 32;
  if (a.pr.D == 64) dq_convert_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(a);
  else if (a.pr.D == 256) dq_convert_kernel<256><<<(unsigned)blocks, 256, 0, st>>>(a);
  else dq_convert_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace lcattn
