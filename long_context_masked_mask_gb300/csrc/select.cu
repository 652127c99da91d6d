// Dynamic block selection: block means of Q and K, pooled scores, and a TopK
// or TopP choice of key blocks per (batch, query head, query block), written
// as the block map that the attention's block-map descriptor consumes.
//
// The selection criterion is the one the paper's peer reviews name for dynamic
// block-sparse attention -- TopK / TopP over pooled Q K^T ("Long-Context
// Attention Benchmark", tomesphere page, section "Peer Reviews") -- and its
// output is the Uniform / Variable Block mask of the xllm-io blog (section
// "注意力掩码模式").  The pages leave the criterion's details open; the readings
// taken here (block means, softmax over the candidates, score-then-index
// ranking, the causal candidate rule) are stated in include/lcattn.h.
//
// Two kernels:
//   pool_kernel    streams Q and K once from HBM (the dominant cost: 2 bytes
//                  per element read, 4 bytes per 128 rows written) and writes
//                  fp32 block means.  One CTA per (batch, block, 8-head slab),
//                  two row groups of 128 threads, 16-byte loads kept eight
//                  deep per thread.
//   select_kernel  one CTA per (batch, head, R consecutive query blocks):
//                  fp32 scores against every key block's mean (read from L2,
//                  stored transposed so that a warp's loads coalesce), a
//                  bitonic sort of 64-bit (score, index) keys per row in
//                  shared memory, then TopK by rank or TopP by a warp scan of
//                  the softmax mass, and a coalesced write of the map rows.
#include <climits>

#include "lcattn_internal.cuh"

namespace lcattn {
namespace {

constexpr int kPoolThreads = 256;   // two row groups of 128 threads
constexpr int kSlabHeads = 8;       // 128 threads x 8 elements = 8 heads x 128
constexpr int kSelThreads = 256;
constexpr int kMaxRows = 8;         // query blocks per select CTA (one warp each for TopP)

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return min(max(x, lo), hi); }

// bf16 pairs in a 32-bit word -> two fp32 values (exact).
__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  #pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(w[i] << 16);
    acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kPoolThreads) pool_kernel(PoolSide qs, PoolSide ks,
                                                            long long q_units) {
  __shared__ float part[128][9];
  long long u = blockIdx.x;
  const bool isq = u < q_units;
  const PoolSide p = isq ? qs : ks;
  if (!isq) u -= q_units;
  const int slab = (int)(u % p.slabs);
  u /= p.slabs;
  const int i = (int)(u % p.nb);
  const int b = (int)(u / p.nb);
  const int t = threadIdx.x & 127;
  const int grp = threadIdx.x >> 7;
  const int h = slab * kSlabHeads + (t >> 4);
  const int e0 = (t & 15) * 8;
  const int lo = clampi(__ldg(p.offs + i), 0, p.S);
  const int hi = clampi(__ldg(p.offs + i + 1), lo, p.S);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (h < p.H) {
    const uint16_t* base = p.x + (int64_t)b * p.sb + (int64_t)h * p.sh + e0;
    int r = lo + grp;
    // Eight loads in flight per thread; rows are summed in increasing order.
    for (; r + 14 < hi; r += 16) {
      uint4 v[8];
      #pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)(r + 2 * k) * p.ss));
      #pragma unroll
      for (int k = 0; k < 8; ++k) add_bf16x8(acc, v[k]);
    }
    for (; r < hi; r += 2)
      add_bf16x8(acc, __ldg(reinterpret_cast<const uint4*>(base + (int64_t)r * p.ss)));
  }
  if (grp == 1) {
    #pragma unroll
    for (int e = 0; e < 8; ++e) part[t][e] = acc[e];
  }
  __syncthreads();
  if (grp == 0 && h < p.H) {
    const int n = hi - lo;
    float m[8];
    #pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = n > 0 ? (acc[e] + part[t][e]) / (float)n : 0.f;
    if (p.transposed) {
      // [B][H][128][nb]: the select kernel's threads (one key block each) then
      // read consecutive addresses.  These 4-byte stores are scattered, but the
      // means are 1/128 of the bytes read.
      float* out = p.out + ((int64_t)b * p.H + h) * kD * p.nb + i;
      #pragma unroll
      for (int e = 0; e < 8; ++e) out[(int64_t)(e0 + e) * p.nb] = m[e];
    } else {
      float4* out = reinterpret_cast<float4*>(p.out + (((int64_t)b * p.H + h) * p.nb + i) * kD + e0);
      out[0] = make_float4(m[0], m[1], m[2], m[3]);
      out[1] = make_float4(m[4], m[5], m[6], m[7]);
    }
  }
}

// Order-preserving map of fp32 to uint32 (larger float -> larger integer).
__device__ __forceinline__ uint32_t ord_of(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_of(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int R = a.R, n2 = a.n2;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);  // [R][n2]
  float* qsm = reinterpret_cast<float*>(keys + (size_t)R * n2);           // [128][kMaxRows]
  int* qend = reinterpret_cast<int*>(qsm + kMaxRows * kD);                // [kMaxRows]
  int* span = qend + kMaxRows;                                            // [1] (+3 pad)
  uint8_t* flags = reinterpret_cast<uint8_t*>(span + 4);                  // [R][nKbp]
  const int nKbp = (a.nKb + 15) & ~15;

  const int tid = threadIdx.x;
  const int nIb = (a.nQb + R - 1) / R;
  int blk = blockIdx.x;
  const int ib = blk % nIb;
  blk /= nIb;
  const int h = blk % a.Hq;
  const int b = blk / a.Hq;
  const int i0 = ib * R;
  const int rows = min(R, a.nQb - i0);
  const int g = h / a.G;
  const int Hkv = a.Hq / a.G;

  const int64_t row0 = ((int64_t)b * a.Hq + h) * a.nQb + i0;  // first map / score row
  for (int x = tid; x < kMaxRows * kD; x += kSelThreads) {
    const int r = x / kD, c = x % kD;
    qsm[c * kMaxRows + r] = r < rows ? a.qbar[(row0 + r) * kD + c] : 0.f;
  }
  if (tid < R) {
    int e = INT_MIN;  // INT_MIN: not a candidate row (past the end, or an empty block)
    if (tid < rows) {
      const int lo = clampi(__ldg(a.q_offs + i0 + tid), 0, a.Sq);
      const int hi = clampi(__ldg(a.q_offs + i0 + tid + 1), lo, a.Sq);
      if (hi > lo) e = hi;
    }
    qend[tid] = e;
  }
  if (tid == 0) *span = 0;
  for (int x = tid; x < R * nKbp; x += kSelThreads) flags[x] = 0;
  __syncthreads();

  // Scores: thread j takes key block j; dot products run over c = 0..127 in
  // order.  k_bar is stored [128][nKb], so a warp's loads are consecutive.
  const float4* q4 = reinterpret_cast<const float4*>(qsm);
  const float* kbar = a.kbar + ((int64_t)b * Hkv + g) * kD * a.nKb;
  for (int j = tid; j < n2; j += kSelThreads) {
    if (j >= a.nKb) {
      for (int r = 0; r < R; ++r) keys[(size_t)r * n2 + j] = 0ull;
      continue;
    }
    const int klo = clampi(__ldg(a.k_offs + j), 0, a.Sk);
    const int khi = clampi(__ldg(a.k_offs + j + 1), klo, a.Sk);
    float acc[kMaxRows];
    #pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.f;
    const float* kp = kbar + j;
    #pragma unroll 8
    for (int c = 0; c < kD; ++c) {
      const float kv = __ldg(kp + (int64_t)c * a.nKb);
      const float4 qa = q4[c * 2], qb = q4[c * 2 + 1];
      acc[0] = fmaf(qa.x, kv, acc[0]);
      acc[1] = fmaf(qa.y, kv, acc[1]);
      acc[2] = fmaf(qa.z, kv, acc[2]);
      acc[3] = fmaf(qa.w, kv, acc[3]);
      acc[4] = fmaf(qb.x, kv, acc[4]);
      acc[5] = fmaf(qb.y, kv, acc[5]);
      acc[6] = fmaf(qb.z, kv, acc[6]);
      acc[7] = fmaf(qb.w, kv, acc[7]);
    }
    bool any = false;
    #pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < R) {
        const float s = acc[r] * a.scale;
        if (a.scores && r < rows) a.scores[(row0 + r) * a.nKb + j] = s;
        const int qe = qend[r];
        const bool cand = qe != INT_MIN && khi > klo && (!a.causal || klo < qe);
        any |= cand;
        keys[(size_t)r * n2 + j] =
            cand ? ((unsigned long long)ord_of(s) << 32) | (uint32_t)(~(uint32_t)j) : 0ull;
      }
    }
    if (any) atomicMax(span, j + 1);
  }
  __syncthreads();

  // Bitonic sort of every row, descending.  A candidate's key is never 0, so
  // candidates come first, in ranking order, then the zeros.
  // Only the first ns keys of each row can be non-zero (ns: a power of two
  // covering the last candidate of any row of this CTA, at least 32), so the
  // sort and the selection run over that prefix; causal rows near the start
  // sort far less than n2.  Every index below is a shift or a mask.
  const int lg2 = __ffs(n2) - 1;
  int lgs = 5;
  while ((1 << lgs) < *span) ++lgs;
  const int ns = 1 << lgs;
  const int lgh = lgs - 1;
  const int pairs = R << lgh;
  for (int lk = 1; lk <= lgs; ++lk) {
    for (int lj = lk - 1; lj >= 0; --lj) {
      const int jj = 1 << lj;
      for (int x = tid; x < pairs; x += kSelThreads) {
        const int r = x >> lgh, pidx = x & ((1 << lgh) - 1);
        const int lo_i = ((pidx >> lj) << (lj + 1)) | (pidx & (jj - 1));
        unsigned long long* row = keys + ((size_t)r << lg2);
        const unsigned long long u = row[lo_i], v = row[lo_i + jj];
        const bool desc = ((lo_i >> lk) & 1) == 0;
        if (desc ? (u < v) : (u > v)) {
          row[lo_i] = v;
          row[lo_i + jj] = u;
        }
      }
      __syncthreads();
    }
  }

  if (a.rule == LCATTN_SELECT_TOPK) {
    const int kk = min(a.top_k, ns);
    for (int x = tid; x < (R << lgs); x += kSelThreads) {
      const int r = x >> lgs, pos = x & (ns - 1);
      const unsigned long long key = keys[((size_t)r << lg2) + pos];
      if (pos < kk && key) flags[r * nKbp + (int)(~(uint32_t)key)] = 1;
    }
  } else {
    // TopP: one warp per row.  Z = sum over candidates of exp(s - s_max)
    // (lane-strided partial sums, then a fixed butterfly); then a running
    // exclusive mass over the ranking, chunk by chunk, keeping a block while
    // the mass before it is below top_p * Z.
    const int warp = tid >> 5, lane = tid & 31;
    for (int r = warp; r < rows; r += kSelThreads / 32) {
      const unsigned long long* row = keys + (size_t)r * n2;
      if (row[0] == 0ull) continue;
      const float s0 = float_of((uint32_t)(row[0] >> 32));
      float z = 0.f;
      for (int pos = lane; pos < ns; pos += 32) {
        const unsigned long long key = row[pos];
        if (key) z += expf(float_of((uint32_t)(key >> 32)) - s0);
      }
      #pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const float pz = a.top_p * z;
      float carry = 0.f;
      for (int base = 0; base < ns; base += 32) {
        const unsigned long long key = row[base + lane];
        const float e = key ? expf(float_of((uint32_t)(key >> 32)) - s0) : 0.f;
        float incl = e;
        #pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const float prev = __shfl_up_sync(0xffffffffu, incl, 1);
        const float before = carry + (lane ? prev : 0.f);
        if (key && before < pz) flags[r * nKbp + (int)(~(uint32_t)key)] = 1;
        carry += __shfl_sync(0xffffffffu, incl, 31);
        const bool done = __any_sync(0xffffffffu, key == 0ull) || !(carry < pz);
        if (done) break;
      }
    }
  }
  __syncthreads();

  for (int x = tid; x < rows * a.nKb; x += kSelThreads) {
    const int r = x / a.nKb, j = x - r * a.nKb;
    a.map[(row0 + r) * a.nKb + j] = flags[r * nKbp + j];
  }
}

}  // namespace

cudaError_t launch_block_pool(const PoolSide& qs, const PoolSide& ks, cudaStream_t st) {
  const long long q_units = (long long)qs.B * qs.nb * qs.slabs;
  const long long k_units = (long long)ks.B * ks.nb * ks.slabs;
  pool_kernel<<<(unsigned)(q_units + k_units), kPoolThreads, 0, st>>>(qs, ks, q_units);
  return cudaGetLastError();
}

size_t select_smem_bytes(int R, int n2, int nKb) {
  const int nKbp = (nKb + 15) & ~15;
  return (size_t)R * n2 * 8 + (size_t)kMaxRows * kD * 4 + kMaxRows * 4 + 16 + (size_t)R * nKbp;
}

void select_geometry(int nKb, int* R, int* n2) {
  int n = 1;
  while (n < nKb) n <<= 1;
  n = n < 32 ? 32 : n;
  int r = kMaxRows;
  while (r > 1 && (size_t)r * n * 8 > 65536) r >>= 1;
  *R = r;
  *n2 = n;
}

cudaError_t launch_block_select(const SelectArgs& a, cudaStream_t st) {
  const size_t smem = select_smem_bytes(a.R, a.n2, a.nKb);
  // Raise the kernel's shared-memory limit only when a call needs more than
  // any call before (so repeated calls, and graph capture, make no such call).
  static size_t smem_set = 48 * 1024;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  const long long ctas = (long long)a.B * a.Hq * ((a.nQb + a.R - 1) / a.R);
  select_kernel<<<(unsigned)ctas, kSelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace lcattn
