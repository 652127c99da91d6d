// Building blocks for context parallelism by Ring P2P (the pages' distributed
// half: "Long-Context Attention Benchmark", xllm-io blog review, section
// "分布式注意力机制" -- K/V shards travel around a ring of devices in several
// point-to-point rounds, each device computes the partial attention of its
// query shard against the K/V shard it holds, and the partial results are
// combined).  These kernels are the per-device pieces:
//   - the mask descriptor of one (query shard, key shard) pair, cut out of the
//     global descriptor;
//   - the merge of a shard pair's partial result (O, LSE) into the running
//     result of the query shard, by log-sum-exp;
//   - the fp32 -> bf16 conversion of accumulated gradients.
// The shard backward itself is the regular backward in accumulate mode
// (bwd.cu).  All kernels are HBM-bound streaming passes.
#include <cuda_bf16.h>

#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

using namespace dev;

int sm_count() {
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  return nsm > 0 ? nsm : 1;
}

__device__ __forceinline__ int shift_clamp(int v, int shift, int limit) {
  const int64_t x = (int64_t)v - shift;
  return (int)(x < 0 ? 0 : (x > limit ? limit : x));
}

// out[b][j] = clamp(in[b][start + j] - shift, 0, limit), componentwise.
__global__ void shard_bounds_kernel(ShardBoundsArgs a) {
  const int64_t total = (int64_t)a.B * a.n;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = t / a.n, j = t - b * a.n;
    const int4 v = __ldg(a.in + b * a.S_in + a.start + j);
    a.out[t] = make_int4(shift_clamp(v.x, a.shift, a.limit), shift_clamp(v.y, a.shift, a.limit),
                         shift_clamp(v.z, a.shift, a.limit), shift_clamp(v.w, a.shift, a.limit));
  }
}

__global__ void shard_offsets_kernel(const int32_t* in, int32_t* out, int n, int shift, int limit) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += gridDim.x * blockDim.x)
    out[i] = shift_clamp(__ldg(in + i), shift, limit);
}

// One warp per (batch, query row, head): merges the shard pair's (O_p, LSE_p)
// into the running (O_acc, LSE_acc):
//   m = max(LSE_acc, LSE_p),  w_acc = exp(LSE_acc - m),  w_p = exp(LSE_p - m),
//   O_acc <- (w_acc O_acc + w_p O_p) / (w_acc + w_p),  LSE_acc <- m + log(w_acc + w_p);
// a row that no shard so far allowed keeps O = 0 and LSE = -inf.
template <int D>
__global__ void lse_merge_kernel(MergeArgs a) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += wstride) {
    const int h = (int)(w % a.pr.Hq);
    const int i = (int)((w / a.pr.Hq) % a.pr.Sq);
    const int b = (int)(w / ((int64_t)a.pr.Hq * a.pr.Sq));
    const int64_t li = ((int64_t)b * a.pr.Hq + h) * a.pr.Sq + i;
    float* acc = a.o_acc + w * D + lane * kPer;  // [B][Sq][Hq][D]: row w
    const __nv_bfloat16* part = reinterpret_cast<const __nv_bfloat16*>(a.o_part) + (int64_t)b * a.p_sb +
                                (int64_t)i * a.p_ss + (int64_t)h * a.p_sh + lane * kPer;
    float op[kPer];
    #pragma unroll
    for (int k = 0; k < kPer; k += 2) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(part + k));
      op[k] = f.x;
      op[k + 1] = f.y;
    }
    const float lp = __ldg(a.lse_part + li);
    float o[kPer];
    float l;
    if (a.first) {
      l = lp;
      #pragma unroll
      for (int k = 0; k < kPer; ++k) o[k] = lp == -INFINITY ? 0.f : op[k];
    } else {
      const float la = a.lse_acc[li];
      const float m = fmaxf(la, lp);
      if (m == -INFINITY) {
        l = -INFINITY;
        #pragma unroll
        for (int k = 0; k < kPer; ++k) o[k] = 0.f;
      } else {
        const float wa = expf(la - m), wp = expf(lp - m);
        const float sum = wa + wp, inv = 1.f / sum;
        l = m + logf(sum);
        #pragma unroll
        for (int k = 0; k < kPer; ++k) o[k] = (wa * acc[k] + wp * op[k]) * inv;
      }
    }
    #pragma unroll
    for (int k = 0; k < kPer; k += 2) *reinterpret_cast<float2*>(acc + k) = make_float2(o[k], o[k + 1]);
    if (lane == 0) a.lse_acc[li] = l;
    if (a.o_out) {
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o_out) + (int64_t)b * a.o_sb +
                           (int64_t)i * a.o_ss + (int64_t)h * a.o_sh + lane * kPer;
      #pragma unroll
      for (int k = 0; k < kPer; k += 2) *reinterpret_cast<uint32_t*>(dst + k) = pack_bf16x2(o[k], o[k + 1]);
    }
  }
}

// fp32 [B][S][H][D] (contiguous) -> bf16 with strides, 8 elements per step.
__global__ void f32_to_bf16_kernel(const float* src, __nv_bfloat16* dst, int64_t B, int64_t S, int64_t H,
                                   int64_t D, int64_t sb, int64_t ss, int64_t sh) {
  const int64_t per_row = D / 8;
  const int64_t n = B * S * H * per_row;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = v % per_row, row = v / per_row;
    const int64_t h = row % H, s = (row / H) % S, b = row / (H * S);
    const float4 x = reinterpret_cast<const float4*>(src + row * D + c * 8)[0];
    const float4 y = reinterpret_cast<const float4*>(src + row * D + c * 8)[1];
    *reinterpret_cast<uint4*>(dst + b * sb + s * ss + h * sh + c * 8) =
        make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
  }
}

unsigned grid_for(int64_t items, int per_block, int cap_per_sm) {
  int64_t blocks = (items + per_block - 1) / per_block;
  const int64_t cap = (int64_t)sm_count() * cap_per_sm;
  if (blocks > cap) blocks = cap;
  return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_shard_bounds(const ShardBoundsArgs& a, cudaStream_t st) {
  shard_bounds_kernel<<<grid_for((int64_t)a.B * a.n, 256, 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_shard_offsets(const int32_t* in, int32_t* out, int n, int shift, int limit,
                                 cudaStream_t st) {
  shard_offsets_kernel<<<grid_for((int64_t)n + 1, 256, 4), 256, 0, st>>>(in, out, n, shift, limit);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.pr.B * a.pr.Sq * a.pr.Hq;
  const unsigned grid = grid_for(rows, 8, 32);  // 8 warps (rows) per 256-thread block
  if (a.pr.D == 64) lse_merge_kernel<64><<<grid, 256, 0, st>>>(a);
  else if (a.pr.D == 128) lse_merge_kernel<128><<<grid, 256, 0, st>>>(a);
  else lse_merge_kernel<256><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t B, int64_t S, int64_t H, int64_t D,
                               int64_t sb, int64_t ss, int64_t sh, cudaStream_t st) {
  f32_to_bf16_kernel<<<grid_for(B * S * H * (D / 8), 256, 32), 256, 0, st>>>(
      src, reinterpret_cast<__nv_bfloat16*>(dst), B, S, H, D, sb, ss, sh);
  return cudaGetLastError();
}

}  // namespace lcattn
