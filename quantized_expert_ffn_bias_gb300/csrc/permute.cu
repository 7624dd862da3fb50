// Batch-union grouping ("25GB RAM runs 744B GLM-5.2" page (pwwt.cn),
// section 3.4): the T*k (token, slot) pairs are grouped by expert so that each
// chosen expert is streamed once for all of its tokens.  Deterministic:
// counting sort by expert id, stable in the flat index t*k + j.
//
// Grid: one CTA per expert.  Every CTA builds the full histogram in shared
// memory (the pair list is small and L2-resident), scans it, and scatters its
// own expert's pairs: each warp counts the matches in a contiguous segment of
// the pairs, and after one block barrier places them with a ballot prefix, so
// the order stays that of t*k + j.  CTA 0 also writes the
// offsets, the list of experts that received tokens (ascending ids) and the
// shared-expert rows.
#include "moe_internal.cuh"

namespace coli {

constexpr int kPermThreads = 256;

__global__ void __launch_bounds__(kPermThreads) permute_kernel(FwdArgs a) {
  __shared__ int hist[kMaxE];
  __shared__ int scan[kMaxE + 1];
  __shared__ int warp_tot[32];
  __shared__ int warp_cnt[kPermThreads / 32];
  __shared__ int total;
  const int E = a.E, P = a.T * a.k, tid = threadIdx.x;
  for (int e = tid; e < E; e += kPermThreads) hist[e] = 0;
  __syncthreads();
#pragma unroll 8
  for (int f = tid; f < P; f += kPermThreads) {
    const int e = a.topk_idx[f];
    if (e < 0 || e >= E) {           // recorded and left out: no row, no output contribution
      if (blockIdx.x == 0) {
        set_status(a.status, COLI_DEV_BAD_EXPERT_ID);
        a.pair_of[f] = -1;
      }
    } else {
      atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  // exclusive scan over E bins, kPermThreads bins per round
  int carry = 0;
  for (int b = 0; b < E; b += kPermThreads) {
    const int e = b + tid;
    const int v = e < E ? hist[e] : 0;
    const int ex = block_exclusive_scan(v, warp_tot, &total);
    if (e < E) scan[e] = carry + ex;
    carry += total;
    __syncthreads();
  }
  if (tid == 0) scan[E] = carry;
  __syncthreads();

  const int me = blockIdx.x;
  if (me < E && hist[me] > 0) {                 // (block-uniform)
    constexpr int kWarps = kPermThreads / 32;
    const int wid = tid >> 5, lane = tid & 31;
    const int seg = ((P + kWarps - 1) / kWarps + 31) & ~31;
    const int s0 = min(P, wid * seg), s1 = min(P, s0 + seg);
    int cnt = 0;
#pragma unroll 8
    for (int f0 = s0; f0 < s1; f0 += 32) {
      const int f = f0 + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, f < s1 && a.topk_idx[f] == me));
    }
    if (lane == 0) warp_cnt[wid] = cnt;
    __syncthreads();
    int pos = scan[me];
    for (int w = 0; w < wid; ++w) pos += warp_cnt[w];
#pragma unroll 8
    for (int f0 = s0; f0 < s1; f0 += 32) {
      const int f = f0 + lane;
      const bool m = f < s1 && a.topk_idx[f] == me;
      const unsigned b = __ballot_sync(0xffffffffu, m);
      if (m) {
        const int at = pos + __popc(b & ((1u << lane) - 1u));
        a.pair_token[at] = f / a.k;
        a.pair_slot[at] = f % a.k;
        a.pair_of[f] = at;
      }
      pos += __popc(b);
    }
  }
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += kPermThreads) a.offsets[e] = scan[e];
    if (tid == 0) a.offsets[E + 1] = P + (a.has_shared ? a.T : 0);
    if (a.has_shared)
      for (int t = tid; t < a.T; t += kPermThreads) a.pair_token[P + t] = t;
    // experts with tokens, ascending
    int ucarry = 0;
    for (int b = 0; b < E; b += kPermThreads) {
      const int e = b + tid;
      const int f = (e < E && hist[e] > 0) ? 1 : 0;
      const int ex = block_exclusive_scan(f, warp_tot, &total);
      if (f) a.unique[ucarry + ex] = e;
      ucarry += total;
      __syncthreads();
    }
    if (tid == 0) {
      a.n_unique[0] = ucarry;
      if (a.has_shared) a.unique[ucarry] = E;
    }
  }
}

cudaError_t launch_permute(const FwdArgs& a, cudaStream_t st) {
  permute_kernel<<<a.E, kPermThreads, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ decode: h -> fixed point / int8 codes
// The SwiGLU outputs of every grouped pair row (valid columns: F, or F_shared
// for the shared expert's rows) in the layout the down kernel reads, one warp
// per block of 32 hidden units: the int4 kernels' 16-bit fixed point, or with
// integer-dot inputs the int8 codes (unpack order for int4, natural for int8).
__global__ void __launch_bounds__(256) quantize_h_kernel(FwdArgs a) {
  griddep_launch_dependents();
  griddep_wait();                  // h of the gate/up kernel
  const int P = a.T * a.k, rows = P + (a.has_shared ? a.T : 0), bpr = a.Fmax / kXqBlock;
  const int lane = threadIdx.x & 31;
  const long long nb = (long long)rows * bpr;
  const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long b = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; b < nb; b += nw) {
    const int r = (int)(b / bpr), c = (int)(b % bpr) * kXqBlock;
    if (c >= (r >= P ? a.Fs : a.F)) continue;          // warp-uniform
    const float v = a.h[(size_t)r * a.Fmax + c + lane];
    uint8_t* dst = reinterpret_cast<uint8_t*>(a.hq + (size_t)r * (a.Fmax / 2)) + (size_t)(c / kXqBlock) * 64;
    int2* qs = a.hqs + (size_t)r * bpr + c / kXqBlock;
    if (!a.idot) warp_quantize_block32(v, dst, qs);
    else if (a.qtype == COLI_Q_INT4_G128) warp_quantize_block32_i8<false>(v, dst, qs);
    else warp_quantize_block32_i8<true>(v, dst, qs);
  }
}

cudaError_t launch_quantize_h(const FwdArgs& a, cudaStream_t st) {
  const int rows = a.T * a.k + (a.has_shared ? a.T : 0);
  const long long warps = (long long)rows * (a.Fmax / kXqBlock);
  int blocks = (int)((warps + 7) / 8);
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  const cudaError_t e = launch_pdl(quantize_h_kernel, dim3(blocks), dim3(256), 0, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------------ debugging aid: the down kernels' input
__global__ void __launch_bounds__(256) debug_hidden_kernel(HiddenView v) {
  const long long n = (long long)v.rows * v.Fmax;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / v.Fmax), c = (int)(i % v.Fmax);
    float val = 0.f;
    if (c < (r >= v.P ? v.Fs : v.F)) {
      if (v.mode == 1) {
        val = v.h[i] / act_prescale(v.qtype, c);
      } else if (v.mode == 4) {
        const int col = v.perm ? ((c & ~7) | ((c & 3) << 1) | ((c >> 2) & 1)) : c;
        val = __half2float(v.hh[(size_t)r * v.Fmax + col]);
      } else {
        const uint8_t* blk = v.hq + (size_t)r * v.Fmax * 2 + (size_t)(c / kXqBlock) * 64;
        const int2 qs = v.hqs[(size_t)r * (v.Fmax / kXqBlock) + c / kXqBlock];
        const int l = c % kXqBlock, j = l & 7, wd = (l >> 3) * 2 + (j & 1);
        const int pos = wd * 4 + (j >> 1);
        int q;
        if (v.mode == 0) q = (int)(int8_t)blk[pos] * 256 + (int)blk[32 + pos];
        else if (v.mode == 2) q = (int)(int8_t)blk[pos];
        else q = (int)(int8_t)blk[l];
        val = __int_as_float(qs.x) * (float)q;
      }
    }
    v.out[i] = val;
  }
}

cudaError_t launch_debug_hidden(const HiddenView& v, cudaStream_t st) {
  const long long n = (long long)v.rows * v.Fmax;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  debug_hidden_kernel<<<blocks, 256, 0, st>>>(v);
  return cudaGetLastError();
}

}  // namespace coli
