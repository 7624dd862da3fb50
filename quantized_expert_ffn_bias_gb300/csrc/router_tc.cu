// Router logits on the tensor cores (bf16 activations, token counts of a
// prefill): z[t][e] = sum_i x[t][i] * Wr[e][i], the routing step of the
// "25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 3.1, with the fp32
// router weights kept exact.
//
// Every fp32 weight splits exactly into three bf16 parts, w = wh + wl + wll
// (wh = bf16(w), wl = bf16(w - wh), wll = w - wh - wl: 8 + 8 + 8 significant
// bits, each residual exact in fp32).  With x in bf16 every product x * part
// is exact in fp32, so three bf16 MMAs with fp32 accumulation sum the same
// exact products as an fp32 GEMM, in another order; single-pass TF32 would
// round the weights to 11 bits and move logits far more than fp32 rounding.
//
// Tiles: 128 tokens (MMA M, TMEM lanes) x 128 experts (MMA N) x one of the
// kRouterKSplit K ranges, one tile per CTA; the K-split partial logits go to
// the workspace's [split][T][E] array, which the top-k kernel sums in split
// order.  A pipeline stage is one 64-element K atom: the x tile and the three
// weight parts (4 x 16 KB, 128-byte swizzle), twelve MMAs per stage.  Warp 0
// loads, warp 1 issues, warps 2..5 read the accumulators back.  All waits are
// bounded.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace coli {

constexpr int kRtM = 128;                    // tokens per tile
constexpr int kRtN = 128;                    // experts per tile
constexpr int kRtStages = 3;
constexpr int kRtAtom = 128 * 128;           // one 64-element K atom of a 128-row tile (bytes)
constexpr int kRtStageBytes = 4 * kRtAtom;   // x, then the three weight parts
constexpr int kRtThreads = 6 * 32;

// w [E * d] fp32 -> out [3][E * d] bf16 (high, middle, low parts), four weights per thread and step
// (n is a multiple of 4: d is a multiple of 128)
__device__ __forceinline__ uint32_t rt_pack(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

__global__ void __launch_bounds__(256) router_split_kernel(const float4* w, long long n4, uint2* out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 v4 = w[i];
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    __nv_bfloat16 h[4], m[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[j] = __float2bfloat16_rn(v[j]);
      const float r1 = v[j] - __bfloat162float(h[j]);   // exact
      m[j] = __float2bfloat16_rn(r1);
      l[j] = __float2bfloat16_rn(r1 - __bfloat162float(m[j]));   // exact: the last 8 bits
    }
    out[i] = make_uint2(rt_pack(h[0], h[1]), rt_pack(h[2], h[3]));
    out[n4 + i] = make_uint2(rt_pack(m[0], m[1]), rt_pack(m[2], m[3]));
    out[2 * n4 + i] = make_uint2(rt_pack(l[0], l[1]), rt_pack(l[2], l[3]));
  }
}

struct RtArgs {
  int T, E, L;            // tokens, experts, K per split
  float* logits;          // [kRouterKSplit][T][E]
  int32_t* status;
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(kRtThreads, 1)
    router_tc_kernel(RtArgs p, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full[kRtStages], empty[kRtStages], acc_full;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtM, ks = blockIdx.y, e0 = blockIdx.z * kRtN;
  const int k0 = ks * p.L, nst = p.L / 64;
  const int ne = min(kRtN, p.E - e0);
  const int N = (ne + 15) & ~15;             // MMA N: the tile's experts rounded up to 16
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(128));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  auto fail_wait = [&]() {
    set_status(p.status, COLI_DEV_WAIT_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      int s = 0;
      bool ok = true;
      for (; s < nst && !*abort_v; ++s) {
        const int st = s % kRtStages;
        if (s >= kRtStages && !mbar_wait(&empty[st], ((s / kRtStages) - 1) & 1, p.wait_ns)) { ok = false; break; }
        uint8_t* dst = smem + (size_t)st * kRtStageBytes;
        mbar_arrive_expect_tx(&full[st], (uint32_t)kRtStageBytes);
        const int kx = k0 + s * 64;
        tma_load_2d_nohint(dst, &xmap, kx, t0, &full[st]);
        for (int q = 0; q < 3; ++q) tma_load_2d_nohint(dst + (1 + q) * kRtAtom, &wmap, kx, q * p.E + e0, &full[st]);
      }
      if (!ok) fail_wait();
      // drain: every issued copy lands before the CTA exits
      for (int j = (s > kRtStages ? s - kRtStages : 0); j < s; ++j)
        mbar_wait(&full[j % kRtStages], (j / kRtStages) & 1, p.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kRtM, N);
      bool ok = true;
      int s = 0;
      for (; s < nst && !*abort_v; ++s) {
        const int st = s % kRtStages;
        if (!mbar_wait_spin(&full[st], (s / kRtStages) & 1, p.wait_ns)) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t xd = umma_desc_sw128(smem_u32(smem + (size_t)st * kRtStageBytes));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            // step kk: 16 elements (32 bytes) of the atom, for the weight part q
            const uint64_t off = (uint64_t)(kk * 2);
            umma_ss(tmem, xd + off, xd + (uint64_t)((1 + q) * kRtAtom >> 4) + off, idesc,
                   (s > 0 || kk > 0 || q > 0) ? 1u : 0u);
          }
        }
        umma_commit(&empty[st]);
      }
      if (!ok) fail_wait();
      umma_commit(&acc_full);                   // also after an abort: the epilogue's wait then ends
      mbar_wait(&acc_full, 0, p.wait_ns);     // the MMAs are complete before tensor memory is freed
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int sp = warp & 3;                  // TMEM sub-partition: lanes 32 sp .. 32 sp + 31
    if (!mbar_wait(&acc_full, 0, p.wait_ns)) {
      fail_wait();
    } else if (!*abort_v) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int t = t0 + sp * 32 + lane;
      float* out = p.logits + ((size_t)ks * p.T + t) * p.E + e0;
      const uint32_t taddr = tmem + ((uint32_t)(sp * 32) << 16);
      for (int c = 0; c < N; c += 16) {
        uint32_t r[16];
        tmem_ld16_issue(taddr + (uint32_t)c, r);
        tmem_ld_wait();
        if (t < p.T) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < ne) out[c + j] = __uint_as_float(r[j]);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128));
  }
}

bool router_tc_applies(const FwdArgs& a) {
  return a.xtype == COLI_X_BF16 && a.T >= kRouterTcMinT && (a.d / kRouterKSplit) % 64 == 0;
}

cudaError_t launch_router_split(const FwdArgs& a, void* wsplit, cudaStream_t st) {
  const long long n4 = (long long)a.E * a.d / 4;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 1216) blocks = 1216;
  router_split_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(a.router_w), n4,
                                              static_cast<uint2*>(wsplit));
  return cudaGetLastError();
}

cudaError_t launch_router_tc(const FwdArgs& a, const void* wsplit, PFN_cuTensorMapEncodeTiled_v12000 encode,
                             cudaStream_t st) {
  CUtensorMap xmap, wmap;
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)a.d, (cuuint64_t)a.T};
    const cuuint64_t gstr[1] = {(cuuint64_t)a.d * 2};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)a.d, (cuuint64_t)(3 * a.E)};
    const cuuint64_t gstr[1] = {(cuuint64_t)a.d * 2};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(wsplit), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  RtArgs p;
  p.T = a.T;
  p.E = a.E;
  p.L = a.d / kRouterKSplit;
  p.logits = a.logits;
  p.status = a.status;
  p.wait_ns = a.wait_ns;
  const size_t smem = (size_t)kRtStages * kRtStageBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.T + kRtM - 1) / kRtM, kRouterKSplit, (a.E + kRtN - 1) / kRtN);
  router_tc_kernel<<<grid, kRtThreads, smem, st>>>(p, xmap, wmap);
  return cudaGetLastError();
}

}  // namespace coli
