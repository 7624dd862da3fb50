// Weighted combine back to token order:
//   out[t] = residual[t] + (sum_j g[t][j] * y[pair_of[t][j]] + y_shared[t])
// summed in slot order j = 0..k-1 (ascending expert id), then the shared
// expert, then the residual.  No atomics: the result is deterministic.
//
// RMSNorm (unit gain) + bf16 rounding for stacked layers.
#include "moe_internal.cuh"

namespace coli {

__global__ void combine_kernel(FwdArgs a) {
  griddep_wait();                  // y of the expert kernels
  const int t = blockIdx.y;
  const int i4 = blockIdx.x * blockDim.x + threadIdx.x;  // float4 index within the row
  if (i4 * 4 >= a.d) return;
  const int P = a.T * a.k;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    // the slot's row indices and rows are loaded first (independent loads), then summed in slot order
    int p[8];
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = j0 + i < a.k ? a.pair_of[(size_t)t * a.k + j0 + i] : -1;
#pragma unroll
    for (int i = 0; i < 8; ++i)   // p < 0: pair left out after a rejected expert id (status word set)
      v[i] = p[i] >= 0 ? *reinterpret_cast<const float4*>(a.y + (size_t)p[i] * a.d + i4 * 4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (p[i] < 0) continue;
      const float g = a.topk_w[(size_t)t * a.k + j0 + i];
      acc.x = fmaf(g, v[i].x, acc.x);
      acc.y = fmaf(g, v[i].y, acc.y);
      acc.z = fmaf(g, v[i].z, acc.z);
      acc.w = fmaf(g, v[i].w, acc.w);
    }
  }
  if (a.has_shared) {
    const float4 v = *reinterpret_cast<const float4*>(a.y + (size_t)(P + t) * a.d + i4 * 4);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  if (a.residual) {
    const float4 r = *reinterpret_cast<const float4*>(a.residual + (size_t)t * a.d + i4 * 4);
    acc.x = r.x + acc.x; acc.y = r.y + acc.y; acc.z = r.z + acc.z; acc.w = r.w + acc.w;
  }
  *reinterpret_cast<float4*>(a.out + (size_t)t * a.d + i4 * 4) = acc;
}

cudaError_t launch_combine(const FwdArgs& a, cudaStream_t st) {
  const int threads = 256;
  dim3 grid((a.d / 4 + threads - 1) / threads, a.T);
  const cudaError_t e = launch_pdl(combine_kernel, grid, dim3(threads), 0, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------------ RMSNorm -> bf16
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__global__ void rmsnorm_bf16_kernel(const float* __restrict__ h, int d, float eps, uint16_t* __restrict__ out) {
  __shared__ float warp_sums[32];
  const int t = blockIdx.x;
  const float* row = h + (size_t)t * d;
  float ss = 0.f;
  for (int i = threadIdx.x * 4; i < d; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
    ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss); ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? warp_sums[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) warp_sums[0] = v;
  }
  __syncthreads();
  const float r = sqrtf(warp_sums[0] / (float)d + eps);
  for (int i = threadIdx.x * 4; i < d; i += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
    ushort4 o;
    o.x = f32_to_bf16_rne(v.x / r);
    o.y = f32_to_bf16_rne(v.y / r);
    o.z = f32_to_bf16_rne(v.z / r);
    o.w = f32_to_bf16_rne(v.w / r);
    *reinterpret_cast<ushort4*>(out + (size_t)t * d + i) = o;
  }
}

cudaError_t launch_rmsnorm_bf16(const float* h, int T, int d, float eps, uint16_t* out, cudaStream_t st) {
  rmsnorm_bf16_kernel<<<T, 256, 0, st>>>(h, d, eps, out);
  return cudaGetLastError();
}

}  // namespace coli
