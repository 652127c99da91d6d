// FP8 forward for sm_103a: the masked attention forward with e4m3 Q, K and V
// (per-tensor descale factors), head dim 128, O in bf16 and LSE in fp32 --
// the fp8-input variant of the operator the pages benchmark ("Long-Context
// Attention Benchmark", xllm-io blog review, sections "密集注意力内核" and
// "稀疏注意力内核").  Both products run as tcgen05 kind::f8f6f4 MMAs with
// fp32 accumulators in TMEM:
//   S = Q8 K8^T                      (A = Q tile, B = K tile, both K-major)
//   O += P8 V8                        (A = P8 from TMEM, B = V^T tile, K-major)
// V^T (key-contiguous rows) is written by a small pre-pass into the
// workspace, so that both operands of the second product are K-major.
// The softmax runs on the exact fp32 logits s * qs * ks * S with the exact
// running row max: P = exp2(t - m) <= 1 is quantized to e4m3 as P * 256 (at
// most 256, inside e4m3's 448) for the PV product, and the row sum l is
// accumulated from the unquantized P.  At the end O = acc * vs / (256 l) and
// LSE = (m + log2 l) ln 2.
//
// One CTA per (query tile, query head, batch), 192 threads: warps 0-3 softmax
// (thread r = query row r = TMEM lane r), warp 4 producer (Q once, K and V^T
// through 2-stage rings), warp 5 TMEM owner and MMA issuer.  80 KB of shared
// memory and 256 TMEM columns (S | O), so two CTAs share an SM and one's
// softmax overlaps the other's products.
#include <cuda_bf16.h>

#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

using namespace dev;

constexpr int kThreads8 = 192;
constexpr int kTile8 = 128 * 128;   // one 128 x 128 e4m3 tile, 128-byte rows
constexpr int kStages8 = 2;
constexpr float kPScale = 256.f;    // P is stored as e4m3(P * 256)
constexpr float kLn2 = 0.6931471805599453f;

struct Fwd8Smem {
  alignas(1024) uint8_t q[kTile8];
  alignas(1024) uint8_t k[kStages8][kTile8];
  alignas(1024) uint8_t vt[kStages8][kTile8];
  uint64_t q_full;
  uint64_t k_full[kStages8], k_empty[kStages8];
  uint64_t v_full[kStages8], v_empty[kStages8];
  uint64_t s_full, p_ready, o_done;
  uint32_t tmem_base;
  int abort_flag;
};

struct Fwd8KernelArgs {
  Fwd8Args a;
};

__device__ __forceinline__ int f8_block_of(const int32_t* offs, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t f8_range_bits(int lo, int hi, int base) {
  const int a = max(lo, base), b = min(hi, base + 32);
  if (b <= a) return 0u;
  const int n = b - a;
  return (n == 32) ? 0xffffffffu : (((1u << n) - 1u) << (a - base));
}

// Allowed-key bits of query row `row` for key tile kt (bit c of word w = key
// kt * 128 + 32 w + c); keys past Sk excluded.
__device__ __forceinline__ void f8_row_mask(const MaskDev& m, const ProblemDev& pr, int b, int h, int row,
                                            int qb_row, bool use_rows, int4 rb, int kt, uint32_t (&mw)[4]) {
  const int k0 = kt * kBN, k1 = min(k0 + kBN, pr.Sk);
  mw[0] = mw[1] = mw[2] = mw[3] = 0u;
  if (row >= pr.Sq) return;
  if (m.kind == LCATTN_MASK_COLBOUNDS) {
    if (use_rows) {
      const int lo0 = max(rb.x, k0) - k0, hi0 = min(rb.y, k1) - k0;
      const int lo1 = max(rb.z, k0) - k0, hi1 = min(rb.w, k1) - k0;
      #pragma unroll
      for (int w = 0; w < 4; ++w) mw[w] = f8_range_bits(lo0, hi0, 32 * w) | f8_range_bits(lo1, hi1, 32 * w);
    } else {
      const int4* cb = m.col_bounds + (int64_t)b * pr.Sk;
      for (int c = 0; c < k1 - k0; ++c) {
        const int4 v = __ldg(cb + k0 + c);
        if ((v.x <= row && row < v.y) || (v.z <= row && row < v.w)) mw[c >> 5] |= 1u << (c & 31);
      }
    }
  } else {
    const uint8_t* map = m.block_map + (((int64_t)b * pr.Hq + h) * m.nQb + qb_row) * (int64_t)m.nKb;
    for (int kb = f8_block_of(m.k_offs, m.nKb, k0); kb < m.nKb; ++kb) {
      const int lo = max(__ldg(m.k_offs + kb), k0);
      if (lo >= k1) break;
      const int hi = min(__ldg(m.k_offs + kb + 1), k1);
      if (hi > lo && __ldg(map + kb)) {
        #pragma unroll
        for (int w = 0; w < 4; ++w) mw[w] |= f8_range_bits(lo - k0, hi - k0, 32 * w);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads8, 2)
fwd8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ Fwd8KernelArgs ka) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Fwd8Args& a = ka.a;
  const ProblemDev& pr = a.pr;
  int32_t* gstatus = a.meta.status;
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(gstatus, 0, LCATTN_ERR_CUDA);
    return;
  }
  Fwd8Smem& sm = *reinterpret_cast<Fwd8Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Unit: (order index, head within the KV group), KV head, batch; longest
  // key lists first (the mask compiler's forward order).
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
    for (int s = 0; s < kStages8; ++s) {
      mbar_init(&sm.k_full[s], 1); mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1); mbar_init(&sm.v_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_ready, 128);
    mbar_init(&sm.o_done, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&sm.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  const int TO = LCATTN_ERR_DEVICE_TIMEOUT;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (n > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmVt);
      }
      __syncwarp();
      mbar_expect_tx_e(&sm.q_full, kTile8);
      tma_load_4d_e(sm.q, &tmQ, &sm.q_full, 0, h, qt * kBM, b);
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int kt = __ldg(lst + j) >> 1;
        const int s = j % kStages8;
        if (j >= kStages8) {
          const bool ok = mbar_wait(&sm.k_empty[s], ((j / kStages8) - 1) & 1, abort_flag, gstatus, TO) &&
                          mbar_wait(&sm.v_empty[s], ((j / kStages8) - 1) & 1, abort_flag, gstatus, TO);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        mbar_expect_tx_e(&sm.k_full[s], kTile8);
        tma_load_4d_e(sm.k[s], &tmK, &sm.k_full[s], 0, g, kt * kBN, b);
        mbar_expect_tx_e(&sm.v_full[s], kTile8);
        tma_load_4d_e(sm.vt[s], &tmVt, &sm.v_full[s], kt * kBN, 0, g, b);
        issued = j + 1;
      }
      int dummy = 0;
      mbar_wait(&sm.q_full, 0, &dummy, gstatus, TO);
      for (int t = max(0, issued - kStages8); t < issued; ++t) {
        mbar_wait(&sm.k_full[t % kStages8], (t / kStages8) & 1, &dummy, gstatus, TO);
        mbar_wait(&sm.v_full[t % kStages8], (t / kStages8) & 1, &dummy, gstatus, TO);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile j: S(j) -> (softmax writes P8 over the S columns) -> O += P8 V(j),
    // then S(j+1) into the same columns (in order after the PV product read them).
    const uint32_t idesc = idesc_e4m3_f32(128, 128);
    const uint32_t tS = tmem, tO = tmem + 128;
    const uint64_t dQ = sdesc_sw128(smem_u32(sm.q), 16, 1024);
    const uint64_t dK = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
    const uint64_t dVt = sdesc_sw128(smem_u32(sm.vt[0]), 16, 1024);
    bool ok = n > 0 && __all_sync(0xffffffffu, mbar_wait(&sm.q_full, 0, abort_flag, gstatus, TO));
    for (int j = 0; ok && j < n; ++j) {
      const int s = j % kStages8;
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[s], (j / kStages8) & 1, abort_flag, gstatus, TO));
      if (!ok) break;
      tc_fence_after();
      {  // S = Q K^T: four k-steps of 32 e4m3 (32 bytes) inside the 128-byte rows
        const uint64_t bk = sdesc_add(dK, s * kTile8);
        mma8_ss_e<0>(tS, dQ, bk, idesc);
        #pragma unroll
        for (int kk = 1; kk < 4; ++kk) mma8_ss_e<1>(tS, sdesc_add(dQ, kk * 32), sdesc_add(bk, kk * 32), idesc);
      }
      tc_commit_e(&sm.k_empty[s]);
      tc_commit_e(&sm.s_full);
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_ready, j & 1, abort_flag, gstatus, TO)) &&
           __all_sync(0xffffffffu, mbar_wait(&sm.v_full[s], (j / kStages8) & 1, abort_flag, gstatus, TO));
      if (!ok) break;
      tc_fence_after();
      {  // O += P8 V: A = P8 from TMEM (4 keys per 32-bit column: 8 columns per k-step)
        const uint64_t bv = sdesc_add(dVt, s * kTile8);
        mma8_ts_er(tO, tS, bv, idesc, j > 0 ? 1u : 0u);
        #pragma unroll
        for (int kk = 1; kk < 4; ++kk) mma8_ts_er(tO, tS + kk * 8, sdesc_add(bv, kk * 32), idesc, 1u);
      }
      tc_commit_e(&sm.v_empty[s]);
      tc_commit_e(&sm.o_done);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = 32 * warp + lane;  // query row within the tile (TMEM lane)
    const int row = qt * kBM + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t tS = tmem + lane_off, tO = tmem + lane_off + 128;
    const float c2 = a.logit_scale_log2;  // scale * qs * ks * log2(e)
    const bool use_rows = a.mask.kind == LCATTN_MASK_COLBOUNDS && a.mask.row_bounds != nullptr;
    int4 rb = make_int4(0, 0, 0, 0);
    int qb_row = 0;
    if (row < pr.Sq) {
      if (use_rows) rb = __ldg(a.mask.row_bounds + (int64_t)b * pr.Sq + row);
      if (a.mask.kind == LCATTN_MASK_BLOCKMAP) qb_row = f8_block_of(a.mask.q_offs, a.mask.nQb, row);
    }
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int e = __ldg(lst + j);
      const int kt = e >> 1;
      const bool masked = (e & 1) != 0 || kt * kBN + kBN > pr.Sk || row >= pr.Sq;
      uint32_t mw[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (masked) f8_row_mask(a.mask, pr, b, h, row, qb_row, use_rows, rb, kt, mw);
      ok = mbar_wait(&sm.s_full, j & 1, abort_flag, gstatus, TO);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // Pass 1: the row max of the logits (log2 domain; masked entries excluded),
      // 32 columns at a time straight from TMEM.
      float mx = -INFINITY;
      #pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t sv[32];
        tmem_ld32(tS + 32 * w, sv);
        tmem_ld_wait();
        #pragma unroll
        for (int c = 0; c < 32; ++c) {
          const bool keep = !masked || ((mw[w] >> c) & 1u);
          mx = keep ? fmaxf(mx, __uint_as_float(sv[c]) * c2) : mx;
        }
      }
      const float m_new = fmaxf(m, mx);
      // Rescale O and l when the row max grows (O holds the products of the
      // previous tiles: wait for the last one first).  The TMEM loads and
      // stores are warp-collective, so the whole warp rescales when any of its
      // rows needs it; rows whose max did not grow scale by exactly 1.
      const bool grow = m_new > m;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        const float alpha = grow ? fast_exp2(m - m_new) : 1.f;
        l *= alpha;
        ok = mbar_wait(&sm.o_done, (j - 1) & 1, abort_flag, gstatus, TO);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        #pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t ov[32];
          tmem_ld32(tO + c, ov);
          tmem_ld_wait();
          #pragma unroll
          for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
          tmem_st32(tO + c, ov);
        }
        tmem_st_wait();
      }
      m = m_new;
      // Pass 2: P = exp2(t - m) (0 for masked entries and for rows with no
      // finite logit yet), the row sum, and e4m3(P * 256) packed 4 keys per
      // column over S's first 32 columns (written after all four loads).
      const float mref = (m == -INFINITY) ? 0.f : m;
      uint32_t pk[32];
      float rs = 0.f;
      #pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t sv[32];
        tmem_ld32(tS + 32 * w, sv);
        tmem_ld_wait();
        #pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float p[4];
          #pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = 4 * c4 + u;
            const bool keep = !masked || ((mw[w] >> c) & 1u);
            p[u] = keep ? fast_exp2(__uint_as_float(sv[c]) * c2 - mref) : 0.f;
            rs += p[u];
          }
          pk[8 * w + c4] = pack_e4m3x4(p[0] * kPScale, p[1] * kPScale, p[2] * kPScale, p[3] * kPScale);
        }
      }
      l += rs;
      // The rescale above (if any) must land before the next product adds to O.
      tmem_st32(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_ready);
    }
    // ---- epilogue: O = acc * vs / (256 l), LSE = (m + log2 l) ln 2
    if (ok) {
      bool have = n > 0;
      if (have) {
        have = __all_sync(0xffffffffu, mbar_wait(&sm.o_done, (n - 1) & 1, abort_flag, gstatus, TO));
        tc_fence_after();
      }
      if (have || n == 0) {
        const bool empty_row = !(l > 0.f);
        const float inv = empty_row ? 0.f : a.v_scale / (kPScale * l);
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.o_sb +
                             (int64_t)row * a.o_ss + (int64_t)h * a.o_sh;
        #pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t ov[32];
          if (n > 0) {
            tmem_ld32(tO + c, ov);
            tmem_ld_wait();
          } else {
            #pragma unroll
            for (int u = 0; u < 32; ++u) ov[u] = 0u;
          }
          if (row < pr.Sq) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
            #pragma unroll
            for (int u = 0; u < 4; ++u)
              d4[u] = make_uint4(pack_bf16x2(__uint_as_float(ov[8 * u]) * inv, __uint_as_float(ov[8 * u + 1]) * inv),
                                 pack_bf16x2(__uint_as_float(ov[8 * u + 2]) * inv, __uint_as_float(ov[8 * u + 3]) * inv),
                                 pack_bf16x2(__uint_as_float(ov[8 * u + 4]) * inv, __uint_as_float(ov[8 * u + 5]) * inv),
                                 pack_bf16x2(__uint_as_float(ov[8 * u + 6]) * inv, __uint_as_float(ov[8 * u + 7]) * inv));
          }
        }
        if (row < pr.Sq)
          a.lse[((int64_t)b * pr.Hq + h) * pr.Sq + row] = empty_row ? -INFINITY : (m + __log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) {
    __syncwarp();
    tmem_dealloc(tmem, 256);
  }
}

// V [B][Sk][Hkv][128] e4m3 -> V^T [B][Hkv][128][Skp] (keys contiguous); keys in
// [Sk, Skp) are written as 0.  One CTA per (64 keys, KV head, batch): 64 x 128
// bytes through shared memory.
__global__ void vt8_kernel(const uint8_t* __restrict__ v, int64_t v_sb, int64_t v_ss, int64_t v_sh,
                           uint8_t* __restrict__ vt, int Sk, int Skp, int Hkv) {
  __shared__ uint8_t t[64][128 + 4];
  const int j0 = blockIdx.x * 64, g = blockIdx.y, b = blockIdx.z;
  for (int idx = threadIdx.x; idx < 64 * 8; idx += blockDim.x) {  // 16 bytes per thread
    const int jj = idx >> 3, c = (idx & 7) * 16;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (j0 + jj < Sk) w = *reinterpret_cast<const uint4*>(v + (int64_t)b * v_sb + (int64_t)(j0 + jj) * v_ss +
                                                          (int64_t)g * v_sh + c);
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(&w);
    #pragma unroll
    for (int u = 0; u < 16; ++u) t[jj][c + u] = wb[u];
  }
  __syncthreads();
  uint8_t* dst = vt + ((int64_t)b * Hkv + g) * 128 * (int64_t)Skp;
  for (int idx = threadIdx.x; idx < 128 * 4; idx += blockDim.x) {  // row d, 16 keys per thread
    const int d = idx >> 2, jj = (idx & 3) * 16;
    if (j0 + jj >= Skp) continue;
    uint32_t w[4];
    #pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = (uint32_t)t[jj + 4 * q][d] | ((uint32_t)t[jj + 4 * q + 1][d] << 8) |
             ((uint32_t)t[jj + 4 * q + 2][d] << 16) | ((uint32_t)t[jj + 4 * q + 3][d] << 24);
    *reinterpret_cast<uint4*>(dst + (int64_t)d * Skp + j0 + jj) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_fwd8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                        const Fwd8Args& a, const uint8_t* v, int64_t v_sb, int64_t v_ss, int64_t v_sh,
                        uint8_t* vt, int Skp, cudaStream_t st) {
  {
    dim3 grid((Skp + 63) / 64, a.pr.Hkv, a.pr.B);
    vt8_kernel<<<grid, 256, 0, st>>>(v, v_sb, v_ss, v_sh, vt, a.pr.Sk, Skp, a.pr.Hkv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  static bool attr_done = false;
  const size_t smem = sizeof(Fwd8Smem);
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(fwd8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  Fwd8KernelArgs ka;
  ka.a = a;
  dim3 grid(a.meta.nQt * a.pr.G, a.pr.Hkv, a.pr.B);
  fwd8_kernel<<<grid, kThreads8, smem, st>>>(tq, tk, tvt, ka);
  return cudaGetLastError();
}

}  // namespace lcattn
