// FP8 forward for sm_103a, its V pre-pass: the masked attention forward with
// e4m3 Q, K and V (per-tensor descale factors), head dim 128, O in bf16 and
// LSE in fp32 -- the fp8-input variant of the operator the pages benchmark
// ("Long-Context Attention Benchmark", xllm-io blog review, sections
// "密集注意力内核" and "稀疏注意力内核").  The forward itself is the persistent
// forward kernel instantiated for e4m3 tiles (both products as tcgen05
// kind::f8f6f4 MMAs, P stored as e4m3 in TMEM); its PV product reads V^T
// (key-contiguous rows) as a K-major operand, which this pre-pass writes into
// the caller's workspace.
#include "lcattn_internal.cuh"

namespace lcattn {
namespace {

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

cudaError_t launch_vt8(const uint8_t* v, int64_t v_sb, int64_t v_ss, int64_t v_sh, uint8_t* vt, int B, int Sk,
                       int Skp, int Hkv, cudaStream_t st) {
  dim3 grid((Skp + 63) / 64, Hkv, B);
  vt8_kernel<<<grid, 256, 0, st>>>(v, v_sb, v_ss, v_sh, vt, Sk, Skp, Hkv);
  return cudaGetLastError();
}

}  // namespace lcattn
