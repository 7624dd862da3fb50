// Router: logits z = x Wr^T (fp32 FMA), s = sigmoid(z), u = s + bias, top-k by u
// (ties -> lower expert id), gate weights g = rho * s / sum(s over the chosen).
//
// "25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 3.1 (sigmoid router,
// 8 of 256) and section 4.3 (the balancing bias steers selection; routing,
// selection and scaling must be reproduced exactly).  Logits stay in fp32 on
// CUDA cores: a TF32 contraction would move scores by ~1e-3 and break exact
// top-k agreement.
#include "moe_internal.cuh"

namespace coli {

// ------------------------------------------------------------------ small-T GEMV
// One warp per (expert, K-slice); partial logits [ks][t][e], summed in ks order
// by the top-k kernel.
template <int NT, int XT>
__global__ void __launch_bounds__(256) router_gemv_kernel(FwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (gw >= a.E * kRouterKSplit) return;
  const int e = gw / kRouterKSplit, ks = gw % kRouterKSplit;
  const int L = a.d / kRouterKSplit;
  const int k0 = ks * L;
  const float* w = a.router_w + (size_t)e * a.d + k0;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 4
  for (int i = lane * 4; i < L; i += 128) {
    const float4 wv = __ldg(reinterpret_cast<const float4*>(w + i));
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < a.T) {
        float x0, x1, x2, x3;
        if (XT == COLI_X_BF16) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2*>(
              static_cast<const uint16_t*>(a.x) + (size_t)t * a.d + k0 + i));
          x0 = __uint_as_float(xv.x << 16);
          x1 = __uint_as_float(xv.x & 0xFFFF0000u);
          x2 = __uint_as_float(xv.y << 16);
          x3 = __uint_as_float(xv.y & 0xFFFF0000u);
        } else {
          const float4 xv = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t * a.d + k0 + i));
          x0 = xv.x; x1 = xv.y; x2 = xv.z; x3 = xv.w;
        }
        acc[t] = fmaf(x0, wv.x, acc[t]);
        acc[t] = fmaf(x1, wv.y, acc[t]);
        acc[t] = fmaf(x2, wv.z, acc[t]);
        acc[t] = fmaf(x3, wv.w, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && t < a.T) a.logits[((size_t)ks * a.T + t) * a.E + e] = v;
  }
}

// ------------------------------------------------------------------ large-T tiled GEMM
// C[t][e] over one K-split: a (16*RM tokens) x 64 (experts) tile per CTA, 256
// threads with RM x 4 outputs each, K in steps of 32.  The next K step's x and
// Wr values are loaded into registers while the current step is computed from
// shared memory (double-buffered, k-major so that each thread reads its
// outputs' operands as two vector loads; columns XOR-swizzled by the k row so
// that the transposing stores are free of bank conflicts).  fp32 FMA in
// ascending k within the split.
constexpr int RB_N = 64, RB_K = 32;

template <int XT, int RM>
__global__ void __launch_bounds__(256) router_gemm_kernel(FwdArgs a) {
  constexpr int RB_M = 16 * RM;
  constexpr int NA = RM / 2;                 // 4-element x loads per thread per K step
  __shared__ __align__(16) float As[2][RB_K][RB_M];
  __shared__ __align__(16) float Bs[2][RB_K][RB_N];
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * RB_N, t0 = blockIdx.y * RB_M, ks = blockIdx.z;
  const int L = a.d / kRouterKSplit, kbeg = ks * L;
  const int tx = tid & 15, ty = tid >> 4;   // outputs: tokens RM*ty.., experts 4*tx..+3
  // global -> register mapping: A rows ra + 32 i (token), 4 k at ca; B row rb (expert), 8 k at cb
  const int ra = tid >> 3, ca = (tid & 7) * 4, rb = tid >> 2, cb = (tid & 3) * 8;
  const bool vb = e0 + rb < a.E;
  const float* wrow = a.router_w + (size_t)(e0 + rb) * a.d + kbeg + cb;
  float4 ar[NA], br0, br1;
  auto load_regs = [&](int kk) {
#pragma unroll
    for (int i = 0; i < NA; ++i) {
      const int t = t0 + ra + 32 * i;
      if (t < a.T) {
        const size_t off = (size_t)t * a.d + kbeg + ca + kk;
        if (XT == COLI_X_BF16) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + off));
          ar[i] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                              __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
        } else {
          ar[i] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + off));
        }
      } else {
        ar[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (vb) {
      br0 = __ldg(reinterpret_cast<const float4*>(wrow + kk));
      br1 = __ldg(reinterpret_cast<const float4*>(wrow + kk + 4));
    } else {
      br0 = br1 = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  // swizzles: A column ^ (k & 28), B column ^ (((k >> 3) & 3) << 3)
  auto store_regs = [&](int buf) {
#pragma unroll
    for (int i = 0; i < NA; ++i) {
      const int sa = (ra + 32 * i) ^ (ca & 28);
      As[buf][ca + 0][sa] = ar[i].x;
      As[buf][ca + 1][sa] = ar[i].y;
      As[buf][ca + 2][sa] = ar[i].z;
      As[buf][ca + 3][sa] = ar[i].w;
    }
    const int sbc = rb ^ (((cb >> 3) & 3) << 3);
    Bs[buf][cb + 0][sbc] = br0.x; Bs[buf][cb + 1][sbc] = br0.y; Bs[buf][cb + 2][sbc] = br0.z;
    Bs[buf][cb + 3][sbc] = br0.w; Bs[buf][cb + 4][sbc] = br1.x; Bs[buf][cb + 5][sbc] = br1.y;
    Bs[buf][cb + 6][sbc] = br1.z; Bs[buf][cb + 7][sbc] = br1.w;
  };
  float acc[RM][4] = {};
  load_regs(0);
  store_regs(0);
  __syncthreads();
  int buf = 0;
  for (int kk = 0; kk < L; kk += RB_K) {
    const bool more = kk + RB_K < L;
    if (more) load_regs(kk + RB_K);
#pragma unroll
    for (int c = 0; c < RB_K; ++c) {
      float av[RM];
      if constexpr (RM == 2) {
        const float2 v = *reinterpret_cast<const float2*>(&As[buf][c][(ty * 2) ^ (c & 28)]);
        av[0] = v.x; av[1] = v.y;
      } else {
        const float4 v = *reinterpret_cast<const float4*>(&As[buf][c][(ty * 4) ^ (c & 28)]);
        av[0] = v.x; av[1] = v.y; av[2] = v.z; av[3] = v.w;
      }
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[buf][c][(tx * 4) ^ (((c >> 3) & 3) << 3)]);
#pragma unroll
      for (int i = 0; i < RM; ++i) {
        acc[i][0] = fmaf(av[i], bv.x, acc[i][0]);
        acc[i][1] = fmaf(av[i], bv.y, acc[i][1]);
        acc[i][2] = fmaf(av[i], bv.z, acc[i][2]);
        acc[i][3] = fmaf(av[i], bv.w, acc[i][3]);
      }
    }
    if (more) {
      store_regs(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }
#pragma unroll
  for (int i = 0; i < RM; ++i) {
    const int t = t0 + ty * RM + i;
    if (t >= a.T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < a.E) a.logits[((size_t)ks * a.T + t) * a.E + e] = acc[i][j];
    }
  }
}

cudaError_t launch_router_logits(const FwdArgs& a, cudaStream_t st) {
  if (a.T <= kDecodeMaxT) {
    const int warps = a.E * kRouterKSplit;
    const int blocks = (warps + 7) / 8;
#define COLI_GEMV(NT)                                                                           \
  if (a.xtype == COLI_X_BF16) router_gemv_kernel<NT, COLI_X_BF16><<<blocks, 256, 0, st>>>(a);   \
  else router_gemv_kernel<NT, COLI_X_F32><<<blocks, 256, 0, st>>>(a);
    if (a.T <= 1) { COLI_GEMV(1) }
    else if (a.T <= 2) { COLI_GEMV(2) }
    else if (a.T <= 4) { COLI_GEMV(4) }
    else { COLI_GEMV(8) }
#undef COLI_GEMV
  } else {
    if (a.T >= 512) {       // 64-token tiles: 4 x 4 outputs per thread
      dim3 grid((a.E + RB_N - 1) / RB_N, (a.T + 63) / 64, kRouterKSplit);
      if (a.xtype == COLI_X_BF16) router_gemm_kernel<COLI_X_BF16, 4><<<grid, 256, 0, st>>>(a);
      else router_gemm_kernel<COLI_X_F32, 4><<<grid, 256, 0, st>>>(a);
    } else {                // 32-token tiles: more CTAs for small T
      dim3 grid((a.E + RB_N - 1) / RB_N, (a.T + 31) / 32, kRouterKSplit);
      if (a.xtype == COLI_X_BF16) router_gemm_kernel<COLI_X_BF16, 2><<<grid, 256, 0, st>>>(a);
      else router_gemm_kernel<COLI_X_F32, 2><<<grid, 256, 0, st>>>(a);
    }
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ top-k
// One warp per token.  Shared memory per warp: u[E], s[E].
constexpr int kTopkWarps = 4;

__device__ __forceinline__ bool better(float ua, int ea, float ub, int eb) {
  return ua > ub || (ua == ub && ea < eb);
}

__device__ __forceinline__ void warp_argmax(float& u, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u2 = __shfl_xor_sync(0xffffffffu, u, o);
    const int e2 = __shfl_xor_sync(0xffffffffu, e, o);
    if (better(u2, e2, u, e)) { u = u2; e = e2; }
  }
}

// Router scores of expert e for token t: s = sigmoid(z) with z the K-split
// partial logits summed in split order, u = s + bias.
__device__ __forceinline__ void router_scores(const FwdArgs& a, int t, int e, float& sv, float& uv) {
  float z = 0.f;
#pragma unroll
  for (int ks = 0; ks < kRouterKSplit; ++ks) z += __ldcg(a.logits + ((size_t)ks * a.T + t) * a.E + e);
  sv = 1.0f / (1.0f + expf(-z));
  uv = sv + __ldg(a.bias + e);
}

// Best (score, expert) among a lane's NV scores (experts lane, lane + 32, ...);
// ties -> lower expert id.
template <int NV>
__device__ __forceinline__ void lane_best(const float (&v)[NV], int lane, int nv, int E, float& bu, int& be) {
  bu = -INFINITY;
  be = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (i < nv && e < E && better(v[i], e, bu, be)) { bu = v[i]; be = e; }
  }
}

// Selection for one token by one warp from its scores in shared memory
// (u, s: [E] each).  Writes topk_idx / topk_w / near_tie and,
// if sel_out is given, the selected ids (ascending) to sel_out[0..k).
// NV = scores per lane (8 keeps them in registers for E <= 256; 32 covers kMaxE).
template <int NV>
__device__ __forceinline__ void topk_select_nv(const FwdArgs& a, int t, float* u, const float* s, int* sel_out) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  // the lane's scores (experts lane, lane+32, ...) in registers; each round the
  // warp takes the best lane candidate and only the winning lane rescans
  const int nv = (E + 31) / 32;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = (i < nv && lane + 32 * i < E) ? u[lane + 32 * i] : -INFINITY;
  float lbu;
  int lbe;
  lane_best(v, lane, nv, E, lbu, lbe);
  int my_sel = -1;          // lane j < k: the j-th pick (by u, descending)
  float kth = 0.f;
  for (int j = 0; j <= k && j < E; ++j) {
    float bu = lbu;
    int be = lbe;
    warp_argmax(bu, be);
    if (j < k) {
      if (lane == j) my_sel = be;
      kth = bu;
      if ((be & 31) == lane) {     // remove the pick from its lane and rescan that lane
#pragma unroll
        for (int i = 0; i < NV; ++i)
          if (i == (be >> 5)) v[i] = -INFINITY;
        lane_best(v, lane, nv, E, lbu, lbe);
      }
    } else {
      const float gap = kth - bu;
      if (lane == 0) a.near_tie[t] = gap < kNearTie ? 1 : 0;
    }
  }
  if (k >= E && lane == 0) a.near_tie[t] = 0;
  // ascending expert-id order: rank of each pick among the picks
  int rank = 0;
  for (int i = 0; i < k; ++i) {
    const int other = __shfl_sync(0xffffffffu, my_sel, i);
    if (lane < k && other < my_sel) ++rank;
  }
  int sorted_e = -1;
  for (int i = 0; i < k; ++i) {
    const int oe = __shfl_sync(0xffffffffu, my_sel, i);
    const int orank = __shfl_sync(0xffffffffu, rank, i);
    if (lane == orank) sorted_e = oe;
  }
  const float my_s = (lane < k) ? s[sorted_e] : 0.f;
  float ssum = 0.f;  // sum in ascending id order
  for (int i = 0; i < k; ++i) ssum += __shfl_sync(0xffffffffu, my_s, i);
  if (lane < k) {
    a.topk_idx[(size_t)t * k + lane] = sorted_e;
    a.topk_w[(size_t)t * k + lane] = a.rho * my_s / ssum;
    if (sel_out) sel_out[lane] = sorted_e;
  }
  __syncwarp();
}

__device__ __forceinline__ void topk_select(const FwdArgs& a, int t, float* u, const float* s, int* sel_out) {
  static_assert(kMaxE == 32 * 32, "lane score array covers kMaxE");
  if (a.E <= 256) topk_select_nv<8>(a, t, u, s, sel_out);
  else topk_select_nv<32>(a, t, u, s, sel_out);
}

// Top-k of one token by one warp.  u, s: this warp's shared scratch [E] each.
__device__ void topk_token(const FwdArgs& a, int t, float* u, float* s) {
  const int lane = threadIdx.x & 31;
#pragma unroll 8
  for (int e = lane; e < a.E; e += 32) router_scores(a, t, e, s[e], u[e]);
  __syncwarp();
  topk_select(a, t, u, s, nullptr);
  // failure-path test: an out-of-range id for the grouping step to reject
  if ((a.inject & COLI_INJECT_BAD_EXPERT_ID) && t == 0 && lane == 0) a.topk_idx[0] = -1;
}

__global__ void __launch_bounds__(kTopkWarps * 32) router_topk_kernel(FwdArgs a) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= a.T) return;
  float* u = sm + (size_t)warp * 2 * a.E;
  topk_token(a, t, u, u + a.E);
}

cudaError_t launch_router_topk(const FwdArgs& a, cudaStream_t st) {
  const int blocks = (a.T + kTopkWarps - 1) / kTopkWarps;
  const size_t smem = (size_t)kTopkWarps * 2 * a.E * sizeof(float);
  router_topk_kernel<<<blocks, kTopkWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ fused decode routing (T <= 8)
// One launch for the whole routing of a decode step:
//   every CTA: its share of the activation pre-scaling (xs) and of the router
//   GEMV (one warp per (expert, K-split), loads issued ahead of the FMAs);
//   the last CTA to finish (atomic ticket on the workspace counter; no waiting)
//   then runs top-k for every token and the batch-union grouping of the
//   T*k <= 256 pairs.
constexpr int kRouteThreads = 256;

template <int NT, int XT>
__global__ void __launch_bounds__(kRouteThreads) route_decode_kernel(FwdArgs a) {
  // dynamic shared memory (last CTA): per token (u[E], s[E])
  extern __shared__ float sm[];
  __shared__ int is_last;
  __shared__ int hist[kDecodeMaxT * kMaxK];   // grouping: first pair of its expert
  __shared__ int ucnt[kDecodeMaxT * kMaxK];   // grouping: pairs of the expert of a first pair
  __shared__ int sidx[kDecodeMaxT * kMaxK];
  const int tid = threadIdx.x, lane = tid & 31;
  griddep_launch_dependents();     // the expert kernel may start its prologue

  // (2) router GEMV partial logits.  The warp's first batch of weight loads is
  //     issued before the activation conversion (1), which runs while they are
  //     in flight; every lane of the warp takes part in (1).
  //     CTA b covers K-split b % kRouterKSplit for experts 8*(b / kRouterKSplit) + warp.
  constexpr int U = 16;
  const int ks_r = blockIdx.x % kRouterKSplit;
  const int e_w = (blockIdx.x / kRouterKSplit) * (kRouteThreads / 32) + (tid >> 5);
  const bool has_row = e_w < a.E;
  const int e_r = has_row ? e_w : 0;
  const int L = a.d / kRouterKSplit, k0 = ks_r * L;
  float* topk_sm = sm;
  const float* wr = a.router_w + (size_t)e_r * a.d + k0;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  float4 wv[U];
  auto load_batch = [&](int base) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 128;
      wv[u] = (has_row && i < L) ? __ldg(reinterpret_cast<const float4*>(wr + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_batch(lane * 4);
  // (1) dequant-GEMV inputs, grid-stride: int4 -> 16-bit fixed point per block
  //     of kXqBlock inputs (one warp per block); int8 -> pre-scaled fp32 + block sums;
  //     integer-dot inputs (both weight types) -> int8 codes per block
  if (a.qtype == COLI_Q_INT4_G128 || a.idot) {
    const int nblk = a.T * a.d / kXqBlock;
    const int nw = gridDim.x * (kRouteThreads / 32);
    for (int b = (blockIdx.x * kRouteThreads + tid) >> 5; b < nblk; b += nw) {
      const int i = b * kXqBlock + lane;
      const float v = XT == COLI_X_BF16 ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.x)[i] << 16)
                                        : static_cast<const float*>(a.x)[i];
      uint8_t* dst = reinterpret_cast<uint8_t*>(a.xq) + (size_t)b * 64;
      if (!a.idot) warp_quantize_block32(v, dst, a.xqs + b);
      else if (a.qtype == COLI_Q_INT4_G128) warp_quantize_block32_i8<false>(v, dst, a.xqs + b);
      else warp_quantize_block32_i8<true>(v, dst, a.xqs + b);
    }
  } else {
    const int n = a.T * a.d;
    for (int i = blockIdx.x * kRouteThreads + tid; i < n; i += gridDim.x * kRouteThreads) {
      const int k = i % a.d;
      float v;
      if (XT == COLI_X_BF16) v = __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.x)[i] << 16);
      else v = static_cast<const float*>(a.x)[i];
      a.xs[i] = v * act_prescale(a.qtype, k);
    }
    const int nb = n / kXsumBlock;   // unscaled sums of x over blocks of 16 inputs
    for (int i = blockIdx.x * kRouteThreads + tid; i < nb; i += gridDim.x * kRouteThreads) {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kXsumBlock; ++j) {
        const int e = i * kXsumBlock + j;
        sum += XT == COLI_X_BF16 ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(a.x)[e] << 16)
                                 : static_cast<const float*>(a.x)[e];
      }
      a.xsum[i] = sum;
    }
  }
  for (int base = lane * 4; base < L; base += 128 * U) {
    if (base != lane * 4) load_batch(base);
    if (!has_row) continue;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t >= a.T) continue;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * 128;
        if (i >= L) continue;
        float x0, x1, x2, x3;
        if (XT == COLI_X_BF16) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) +
                                                                (size_t)t * a.d + k0 + i));
          x0 = __uint_as_float(xv.x << 16);
          x1 = __uint_as_float(xv.x & 0xFFFF0000u);
          x2 = __uint_as_float(xv.y << 16);
          x3 = __uint_as_float(xv.y & 0xFFFF0000u);
        } else {
          const float4 xv =
              __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t * a.d + k0 + i));
          x0 = xv.x; x1 = xv.y; x2 = xv.z; x3 = xv.w;
        }
        acc[t] = fmaf(x0, wv[u].x, acc[t]);
        acc[t] = fmaf(x1, wv[u].y, acc[t]);
        acc[t] = fmaf(x2, wv[u].z, acc[t]);
        acc[t] = fmaf(x3, wv[u].w, acc[t]);
      }
    }
  }
  if (has_row) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t < a.T) a.logits[((size_t)ks_r * a.T + t) * a.E + e_r] = v;
    }
  }
  // (3) ticket: the last CTA to arrive does the rest
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(a.status + 1, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // (4) top-k: every thread loads scores (all loads independent), then one warp per token selects
  for (int i = tid; i < a.T * a.E; i += kRouteThreads) {
    const int t = i / a.E, e = i - t * a.E;
    float* u = topk_sm + (size_t)t * 2 * a.E;
    router_scores(a, t, e, u[a.E + e], u[e]);
  }
  __syncthreads();
  {
    const int warp = tid >> 5;
    for (int t = warp; t < a.T; t += kRouteThreads / 32) {
      float* u = topk_sm + (size_t)t * 2 * a.E;
      topk_select(a, t, u, u + a.E, sidx + t * a.k);
    }
  }
  __syncthreads();
  const int E = a.E, P = a.T * a.k;
  // a failure-path test plants an out-of-range id here; any id outside [0, E) is recorded in the
  // status word and mapped to E, which sorts after every expert and is left out of the grouping
  if ((a.inject & COLI_INJECT_BAD_EXPERT_ID) && tid == 0) sidx[0] = -1;
  __syncthreads();
  for (int f = tid; f < P; f += kRouteThreads) {
    if (sidx[f] < 0 || sidx[f] >= E) {
      set_status(a.status, COLI_DEV_BAD_EXPERT_ID);
      sidx[f] = E;
    }
  }
  __syncthreads();
  // (5) grouping of the P = T*k <= 256 pairs (stable counting sort by expert id),
  //     by direct counting over the pairs: position of pair f = pairs with a lower
  //     expert id, plus earlier pairs of the same expert
  for (int f = tid; f < P; f += kRouteThreads) {
    const int e = sidx[f];
    if (e == E) {                    // left out: no row, no output contribution
      a.pair_of[f] = -1;
      hist[f] = 0;
      continue;
    }
    int pos = 0, first = 1;
    for (int g = 0; g < P; ++g) {
      const int eg = sidx[g];
      pos += (eg < e) || (eg == e && g < f);
      first &= !(eg == e && g < f);
    }
    a.pair_token[pos] = f / a.k;
    a.pair_slot[pos] = f % a.k;
    a.pair_of[f] = pos;
    hist[f] = first;                 // first pair (in flat order) of its expert
  }
  for (int e = tid; e <= E; e += kRouteThreads) {
    int below = 0;
    for (int g = 0; g < P; ++g) below += sidx[g] < e;
    a.offsets[e] = below;
  }
  if (tid == 0) a.offsets[E + 1] = P + (a.has_shared ? a.T : 0);
  if (a.has_shared)
    for (int t = tid; t < a.T; t += kRouteThreads) a.pair_token[P + t] = t;
  __syncthreads();
  // experts with tokens, ascending: rank of each expert's first pair among the
  // first pairs.  utab gets (slot, first pair row, pairs) per entry for the
  // dequant-GEMV kernels, ordered by pairs, most first (ties: ascending id):
  // units are dealt in utab order, so the experts that take several passes
  // start in the first round instead of lengthening the last one
  for (int f = tid; f < P; f += kRouteThreads) {
    int cnt = 0;
    if (hist[f]) {
      const int e = sidx[f];
      for (int g = 0; g < P; ++g) cnt += sidx[g] == e;
    }
    ucnt[f] = cnt;                   // pairs of the expert whose first pair f is (0: not a first pair)
  }
  __syncthreads();
  for (int f = tid; f < P; f += kRouteThreads) {
    if (!hist[f]) continue;
    const int e = sidx[f], cnt = ucnt[f];
    int r = 0, below = 0, ro = 0;
    for (int g = 0; g < P; ++g) {
      r += hist[g] && sidx[g] < e;
      below += sidx[g] < e;
      ro += hist[g] && (ucnt[g] > cnt || (ucnt[g] == cnt && sidx[g] < e));
    }
    a.unique[r] = e;
    a.utab[ro] = make_int4(e, below, cnt, 0);
  }
  if (tid == 0) {
    int nu = 0;
    for (int g = 0; g < P; ++g) nu += hist[g];
    a.n_unique[0] = nu;
    if (a.has_shared) {
      a.unique[nu] = E;
      a.utab[nu] = make_int4(E, P, a.T, 0);
    }
    a.status[1] = 0;
  }
}

cudaError_t launch_route_decode(const FwdArgs& a, cudaStream_t st) {
  const int blocks = ((a.E + kRouteThreads / 32 - 1) / (kRouteThreads / 32)) * kRouterKSplit;
  const size_t smem = (size_t)a.T * 2 * a.E * sizeof(float);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
#define COLI_ROUTE(NT)                                                                                    \
  {                                                                                                       \
    auto kern = a.xtype == COLI_X_BF16 ? route_decode_kernel<NT, COLI_X_BF16> : route_decode_kernel<NT, COLI_X_F32>; \
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);   \
    if (e != cudaSuccess) return e;                                                                       \
    kern<<<blocks, kRouteThreads, smem, st>>>(a);                                                         \
  }
  if (a.T <= 1) COLI_ROUTE(1)
  else if (a.T <= 2) COLI_ROUTE(2)
  else if (a.T <= 4) COLI_ROUTE(4)
  else COLI_ROUTE(8)
#undef COLI_ROUTE
  return cudaGetLastError();
}

}  // namespace coli
