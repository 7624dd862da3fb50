// Key selection of sparse attention: the "lightning indexer" scores and its
// top-k ("25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 3.3: every layer
// keeps the top-2048 causal keys; section 4.4: a light indexer scores the
// earlier keys and the top-k entries are selected, the indexer itself doing
// the scoring and the top-k).  The scoring formula is that of the DeepSeek-V3.2
// indexer the page cites:
//   I[t][s] = sum_{j < H} w[t][j] * relu(q[t][j] . k[s])
// for the keys s <= pos0 + t the query at position pos0 + t sees.
//
// Scores: a dense contraction of the keys [L][128] with the queries' heads
// [64 T][128] on the 5th-generation tensor cores (bf16 operands staged by TMA
// in shared memory, fp32 accumulators in tensor memory), one CTA per SM over
// tiles of 128 keys.  Warp 0 loads, warp 1 issues the MMAs (M = 128 keys,
// N = 64 heads x up to 4 queries, K = 128 in eight steps), warps 2..5 read the
// accumulators back and form relu, the head-weighted sum (heads in ascending
// order) and the causal mask.  Double-buffered accumulators let the MMAs of one
// tile overlap the epilogue of the previous one.  All waits are bounded.
//
// Top-k: the score kernel also counts every visible score in a 65536-bin
// histogram of the top 16 bits of its order-preserving integer image.  A
// marking kernel (16 CTAs per query at 65,536 keys) finds the bin of the
// topk-th score from it, sets the bits of the keys above that bin in a key
// bitmask and gathers the keys in it; one CTA per query then ranks those
// exactly (score, then key index) and writes the bitmask out in key order.
#include "moe_internal.cuh"

namespace coli {

constexpr int kIxKeys = 128;        // keys per tile (MMA M, TMEM lanes)
constexpr int kIxD = 128;           // head dimension (two 64-element swizzle atoms)
constexpr int kIxHeads = 64;        // heads per query
constexpr int kIxQMax = 4;          // queries per launch (MMA N = 64 * queries <= 256)
constexpr int kIxStages = 4;
constexpr int kIxThreads = 6 * 32;
constexpr int kIxAtomKeys = kIxKeys * 128;            // bytes of one 64-element atom of a key tile
constexpr int kIxStageBytes = 2 * kIxAtomKeys;        // 32 KB
constexpr int kIxTopkThreads = 1024;

struct IxArgs {
  int T, L, pos0;
  const float* w;        // [T][64] head weights of this launch's queries
  float* scores;         // [T][ls]
  int ls;
  uint32_t* hist;        // [T][65536]: visible scores per top 16 bits of their integer image (cleared before)
  uint32_t* chist;       // [T][2048]: the same per top 11 bits (cleared before)
  int32_t* status;
  unsigned long long wait_ns;
};

// Order-preserving integer image of an fp32 value.
__device__ __forceinline__ uint32_t ix_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ix_unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint64_t ix_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused for a K-major 128-byte atom)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: bf16 A and B, both K-major, fp32 accumulate.
__device__ __forceinline__ uint32_t ix_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void ix_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void ix_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void ix_tma_load(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kIxThreads, 1)
    indexer_scores_kernel(IxArgs p, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t full[kIxStages], empty[kIxStages], q_full, acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ float ws[kIxQMax * kIxHeads];
  __shared__ uint32_t ch[kIxQMax][1024];   // this CTA's share of the coarse histogram, two 16-bit counts a word
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem + kIxStages * kIxStageBytes;   // queries: two atoms of N rows x 128 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = kIxHeads * p.T;
  const int n_tiles = (p.L + kIxKeys - 1) / kIxKeys;
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kIxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < p.T * kIxHeads; i += blockDim.x) ws[i] = p.w[i];
  for (int i = threadIdx.x; i < p.T * 1024; i += blockDim.x) (&ch[0][0])[i] = 0u;
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(512));
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
      mbar_arrive_expect_tx(&q_full, (uint32_t)(2 * N * 128));
      for (int at = 0; at < 2; ++at) ix_tma_load(qs + at * N * 128, &qmap, at * 64, 0, &q_full);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++it) {
        const int s = it % kIxStages;
        if (it >= kIxStages && !mbar_wait(&empty[s], ((it / kIxStages) - 1) & 1, p.wait_ns)) { ok = false; break; }
        uint8_t* st = smem + (size_t)s * kIxStageBytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kIxStageBytes);
        for (int at = 0; at < 2; ++at) ix_tma_load(st + at * kIxAtomKeys, &kmap, at * 64, t * kIxKeys, &full[s]);
      }
      if (!ok) fail_wait();
      // drain: every issued copy lands before the CTA exits
      mbar_wait(&q_full, 0, p.wait_ns);
      for (int j = (it > kIxStages ? it - kIxStages : 0); j < it; ++j)
        mbar_wait(&full[j % kIxStages], (j / kIxStages) & 1, p.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ix_idesc_bf16(kIxKeys, N);
      bool ok = mbar_wait_spin(&q_full, 0, p.wait_ns);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t qd = ix_desc_sw128(smem_u32(qs));
      const uint64_t q_atom = (uint64_t)((N * 128) >> 4);
      int i = 0;
      for (int t = blockIdx.x; ok && t < n_tiles && !*abort_v; t += gridDim.x, ++i) {
        const int s = i % kIxStages, acc = i & 1;
        if (!mbar_wait_spin(&full[s], (i / kIxStages) & 1, p.wait_ns)) { ok = false; break; }
        if (i >= 2 && !mbar_wait_spin(&acc_empty[acc], ((i >> 1) - 1) & 1, p.wait_ns)) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t kd = ix_desc_sw128(smem_u32(smem + (size_t)s * kIxStageBytes));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // step kk: 16 elements (32 bytes) of atom kk / 4 of both operands
          const uint64_t off = (uint64_t)((kk & 3) * 2);
          const uint64_t a = kd + off + (kk >= 4 ? (uint64_t)(kIxAtomKeys >> 4) : 0);
          const uint64_t b = qd + off + (kk >= 4 ? q_atom : 0);
          ix_mma(tmem + (uint32_t)(acc * N), a, b, idesc, kk > 0 ? 1u : 0u);
        }
        ix_commit(&empty[s]);
        ix_commit(&acc_full[acc]);
      }
      if (!ok) fail_wait();
      // the last accumulators must be complete before the CTA frees tensor memory
      if (i > 0) mbar_wait(&acc_full[(i - 1) & 1], ((i - 1) >> 1) & 1, p.wait_ns);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int sp = warp & 3;                  // TMEM sub-partition: lanes 32 sp .. 32 sp + 31
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles && !*abort_v; t += gridDim.x, ++i) {
      const int acc = i & 1;
      if (!mbar_wait(&acc_full[acc], (i >> 1) & 1, p.wait_ns)) { fail_wait(); break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int s = t * kIxKeys + sp * 32 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(sp * 32) << 16) + (uint32_t)(acc * N);
      for (int q = 0; q < p.T; ++q) {
        // the query's 64 head columns: four 16-column loads in flight, one wait
        uint32_t r[kIxHeads];
#pragma unroll
        for (int c = 0; c < kIxHeads / 16; ++c)
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
              : "=r"(r[c * 16 + 0]), "=r"(r[c * 16 + 1]), "=r"(r[c * 16 + 2]), "=r"(r[c * 16 + 3]),
                "=r"(r[c * 16 + 4]), "=r"(r[c * 16 + 5]), "=r"(r[c * 16 + 6]), "=r"(r[c * 16 + 7]),
                "=r"(r[c * 16 + 8]), "=r"(r[c * 16 + 9]), "=r"(r[c * 16 + 10]), "=r"(r[c * 16 + 11]),
                "=r"(r[c * 16 + 12]), "=r"(r[c * 16 + 13]), "=r"(r[c * 16 + 14]), "=r"(r[c * 16 + 15])
              : "r"(taddr + (uint32_t)(q * kIxHeads + c * 16)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < kIxHeads; ++j) sum = fmaf(ws[q * kIxHeads + j], fmaxf(__uint_as_float(r[j]), 0.f), sum);
        const bool vis = s < p.L && s <= p.pos0 + q;
        if (s < p.L) p.scores[(size_t)q * p.ls + s] = vis ? sum : -INFINITY;
        // the selection's histograms: top 16 bits of the score's order-preserving image (global) and
        // top 11 bits (this CTA's share, added to the global one at the end)
        if (vis) {
          const uint32_t key = ix_key(sum);
          atomicAdd(p.hist + ((size_t)q << 16) + (key >> 16), 1u);
          atomicAdd(&ch[q][key >> 22], 1u << (16 * ((key >> 21) & 1)));   // < 2^16 keys per CTA and query
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
  for (int i = threadIdx.x; i < p.T * 1024; i += blockDim.x) {
    const uint32_t v = (&ch[0][0])[i];
    if (v & 0xFFFFu) atomicAdd(p.chist + 2 * i, v & 0xFFFFu);
    if (v >> 16) atomicAdd(p.chist + 2 * i + 1, v >> 16);
  }
}

// ------------------------------------------------------------------ top-k (one CTA per query)

constexpr int kIxMaxKeys = 1 << 17;      // keys one selection serves (the key bitmask lives in shared memory)
constexpr int kIxCand = 2048;            // candidates of the boundary bin kept in shared memory
constexpr int kIxBatch = 16;             // rounds of scores loaded ahead in the selection passes

// Bin (of nb) of the rem-th largest element and the rank `rem` within it, from a histogram in shared
// memory.  All threads call it; the result is in *s_bin / *s_rem after it returns.
__device__ __forceinline__ void ix_find_bin(const int* hist, int nb, int rem, int* warp_tot, int* total,
                                            int* s_bin, int* s_rem) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int per = nb / nthr > 0 ? nb / nthr : 1;   // bins per thread, from the top down
  const int first = nb - 1 - tid * per;
  int c = 0;
  if (tid * per < nb)
    for (int j = 0; j < per; ++j) c += hist[first - j];
  const int above = block_exclusive_scan(c, warp_tot, total);
  if (tid * per < nb && above < rem && rem <= above + c) {
    int cum = above;
    for (int j = 0; j < per; ++j) {
      const int b = first - j;
      if (cum + hist[b] >= rem) {
        *s_bin = b;
        *s_rem = rem - cum;
        break;
      }
      cum += hist[b];
    }
  }
  __syncthreads();
}

// Warp-aggregated shared-memory histogram increment: lanes with the same bin add once.
__device__ __forceinline__ void ix_hist_add(int* hist, int bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

constexpr int kIxChunk = 4096;           // keys per CTA of the marking kernel
constexpr int kIxMarkThreads = 256;

struct IxSel {
  const float* scores;     // [T][ls]
  int ls, L, pos0, topk;
  const uint32_t* hist;    // [T][65536]
  const uint32_t* chist;   // [T][2048]
  uint32_t* bits;          // [T][ws_words] selected-key bitmask (keys above the boundary bin)
  int ws_words;
  float* cand_val;         // [T][kIxCand] boundary-bin keys
  int* cand_idx;
  int* cand_n;             // [T] (cleared before the scores are computed)
  int32_t* out;            // [T][topk]
};

__device__ __forceinline__ int ix_visible(const IxSel& p, int q) {
  const long long v = (long long)p.pos0 + q + 1;   // keys s <= pos0 + q, s < L
  return v < p.L ? (int)v : p.L;
}

// Bin of the topk-th largest score: the query's 2048-bin histogram (top 11 bits of the integer image),
// scanned from the top by the whole CTA, names the coarse bin; warp 0 then scans the 32 fine bins (top 16
// bits) inside it.  (bin, rank within it, keys in it) land in shared memory.
__device__ __forceinline__ void ix_boundary(const uint32_t* gh, const uint32_t* gch, int topk, int* warp_tot,
                                            int* total, int* s_bin, int* s_rem, int* s_cnt, int* s_run) {
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
  const int per = 2048 / nthr;             // coarse bins per thread (8 or 2)
  const int top = 2047 - tid * per;
  int h[8];
  int c = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {            // h[i]: bin top - i
    h[i] = i < per ? (int)__ldcg(gch + top - i) : 0;
    c += h[i];
  }
  const int above = block_exclusive_scan(c, warp_tot, total);
  if (above < topk && topk <= above + c) {
    int cum = above;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < per && cum + h[i] >= topk) {
        s_run[0] = top - i;                // coarse bin
        s_run[1] = cum;                    // keys in higher coarse bins
        break;
      }
      cum += h[i];
    }
  }
  __syncthreads();
  if (tid < 32) {
    const int cb = s_run[0];
    const int fb = cb * 32 + 31 - lane;    // lane 0: the highest fine bin of the coarse bin
    const int hf = (int)__ldcg(gh + fb);
    int inc = hf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    const int cum = s_run[1] + inc - hf;
    if (cum < topk && topk <= cum + hf) {
      *s_bin = fb;
      *s_rem = topk - cum;
      *s_cnt = hf;
    }
  }
  __syncthreads();
}

// Grid (chunks of kIxChunk keys, queries): keys above the boundary bin set their bit in the query's
// bitmask (warp ballots), keys in it are appended to the query's candidate list (warp-aggregated).
__global__ void __launch_bounds__(kIxMarkThreads) indexer_mark_kernel(IxSel p) {
  __shared__ int warp_tot[32];
  __shared__ int total, s_bin, s_rem, s_cnt, s_run[2];
  const int q = blockIdx.y, lane = threadIdx.x & 31;
  const int vis = ix_visible(p, q);
  const int k0 = blockIdx.x * kIxChunk;
  if (vis <= p.topk || k0 >= vis) return;          // (block-uniform)
  ix_boundary(p.hist + ((size_t)q << 16), p.chist + ((size_t)q << 11), p.topk, warp_tot, &total, &s_bin, &s_rem,
              &s_cnt, s_run);
  const uint32_t bin = (uint32_t)s_bin;
  const bool keep = s_cnt <= kIxCand;               // otherwise the finishing kernel takes the long way
  const float* sc = p.scores + (size_t)q * p.ls;
  uint32_t* bits = p.bits + (size_t)q * p.ws_words;
  constexpr int kPer = kIxChunk / kIxMarkThreads;
  float vb[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int s = k0 + i * kIxMarkThreads + threadIdx.x;
    vb[i] = s < vis ? sc[s] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int s = k0 + i * kIxMarkThreads + threadIdx.x;
    const bool valid = s < vis;
    const uint32_t b = valid ? ix_key(vb[i]) >> 16 : 0u;
    const unsigned word = __ballot_sync(0xffffffffu, valid && b > bin);
    if (lane == 0 && s < vis) bits[s >> 5] = word;
    const unsigned cm = keep ? __ballot_sync(0xffffffffu, valid && b == bin) : 0u;
    if (cm) {
      int base = 0;
      if (lane == __ffs(cm) - 1) base = atomicAdd(p.cand_n + q, __popc(cm));
      base = __shfl_sync(0xffffffffu, base, __ffs(cm) - 1);
      if (valid && b == bin) {
        const int c = base + __popc(cm & ((1u << lane) - 1u));
        if (c < kIxCand) {   // the bin holds s_cnt <= kIxCand keys in all
          p.cand_val[(size_t)q * kIxCand + c] = vb[i];
          p.cand_idx[(size_t)q * kIxCand + c] = s;
        }
      }
    }
  }
}

// One CTA per query: the boundary-bin candidates ranked exactly (score descending, key ascending), the
// first `rem` added to the bitmask, and the bitmask written out in key order.  A boundary bin with more
// keys than the candidate list holds (many equal or near-equal scores) takes the long way: an exact
// radix select on the integer image (11 + 11 + 10 bits over three passes) gives the threshold, and one
// marking pass takes the keys above it and, in key order, the first keys equal to it.
__global__ void __launch_bounds__(kIxTopkThreads) indexer_finish_kernel(IxSel p) {
  __shared__ uint32_t bits[kIxMaxKeys / 32];
  __shared__ int hist[2048];
  __shared__ float cand_val[kIxCand];
  __shared__ int cand_idx[kIxCand];
  __shared__ int warp_tot[32];
  __shared__ int total, s_bin, s_rem, s_cnt, s_eq, s_run[2];
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
  const int q = blockIdx.x;
  const float* sc = p.scores + (size_t)q * p.ls;
  int32_t* o = p.out + (size_t)q * p.topk;
  const int vis = ix_visible(p, q), topk = p.topk;
  if (vis <= topk) {
    for (int i = tid; i < topk; i += nthr) o[i] = i < vis ? i : -1;
    return;
  }
  const int nwords = (vis + 31) / 32;
  const int rounds = (vis + nthr - 1) / nthr;
  ix_boundary(p.hist + ((size_t)q << 16), p.chist + ((size_t)q << 11), topk, warp_tot, &total, &s_bin, &s_rem,
              &s_cnt, s_run);
  int rem = s_rem;
  if (s_cnt <= kIxCand) {
    const uint32_t* gbits = p.bits + (size_t)q * p.ws_words;
    for (int i = tid; i < nwords; i += nthr) bits[i] = __ldcg(gbits + i);
    const int nc = s_cnt;
    for (int c = tid; c < nc; c += nthr) {
      cand_val[c] = __ldcg(p.cand_val + (size_t)q * kIxCand + c);
      cand_idx[c] = __ldcg(p.cand_idx + (size_t)q * kIxCand + c);
    }
    __syncthreads();
    for (int c = tid; c < nc; c += nthr) {
      const float v = cand_val[c];
      const int si = cand_idx[c];
      int rank = 0;
      for (int e = 0; e < nc; ++e) rank += cand_val[e] > v || (cand_val[e] == v && cand_idx[e] < si);
      if (rank < rem) atomicOr(&bits[si >> 5], 1u << (si & 31));
    }
    __syncthreads();
  } else {
    for (int i = tid; i < nwords; i += nthr) bits[i] = 0u;
    uint32_t prefix = 0, mask = 0;
    rem = topk;
    for (int pass = 0; pass < 3; ++pass) {
      const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0), w = pass == 2 ? 10 : 11;
      const uint32_t bm = (1u << w) - 1u;
      __syncthreads();
      for (int b = tid; b < 2048; b += nthr) hist[b] = 0;
      __syncthreads();
      for (int r = 0; r < rounds; ++r) {
        const int s = r * nthr + tid;
        const uint32_t u = s < vis ? ix_key(sc[s]) : 0u;
        const bool hit = s < vis && (u & mask) == prefix;
        ix_hist_add(hist, hit ? (int)((u >> sh) & bm) : 0, hit);
      }
      __syncthreads();
      ix_find_bin(hist, 1 << w, rem, warp_tot, &total, &s_bin, &s_rem);
      prefix |= (uint32_t)s_bin << sh;
      mask |= bm << sh;
      rem = s_rem;
    }
    if (tid == 0) s_eq = 0;
    __syncthreads();
    for (int r = 0; r < rounds; ++r) {
      const int s = r * nthr + tid;
      const bool valid = s < vis;
      const uint32_t u = valid ? ix_key(sc[s]) : 0u;
      const bool eq = valid && u == prefix;
      const int before = block_exclusive_scan(eq ? 1 : 0, warp_tot, &total);   // equal keys earlier in the round
      const bool take = valid && (u > prefix || (eq && s_eq + before < rem));
      const unsigned word = __ballot_sync(0xffffffffu, take);
      if (lane == 0 && s < vis) bits[s >> 5] = word;
      __syncthreads();
      if (tid == 0) s_eq += total;
      __syncthreads();
    }
  }
  // emit in key order: each thread a contiguous run of words
  const int wpt = (nwords + nthr - 1) / nthr;
  const int w0 = tid * wpt, w1 = min(nwords, w0 + wpt);
  int cnt = 0;
  for (int i = w0; i < w1; ++i) cnt += __popc(bits[i]);
  int pos = block_exclusive_scan(cnt, warp_tot, &total);
  for (int i = w0; i < w1; ++i) {
    uint32_t m = bits[i];
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1;
      if (pos < topk) o[pos] = i * 32 + b;   // exactly topk bits are set; the bound keeps a miscount inside
      ++pos;
    }
  }
}

// ------------------------------------------------------------------ host side

cudaError_t launch_indexer(const IndexerCall& c, cudaStream_t st, int num_sms) {
  cudaError_t e = c.steps & 1 ? launch_indexer_scores(c, st, num_sms) : cudaSuccess;
  if (e == cudaSuccess && (c.steps & 2)) {
    IxSel p;
    p.scores = c.scores;
    p.ls = c.L;
    p.L = c.L;
    p.pos0 = c.pos0;
    p.topk = c.topk;
    p.hist = c.hist;
    p.chist = c.chist;
    p.bits = c.sel_bits;
    p.ws_words = (c.L + 31) / 32;
    p.cand_val = c.cand_val;
    p.cand_idx = c.cand_idx;
    p.cand_n = c.cand_n;
    p.out = c.out;
    indexer_mark_kernel<<<dim3((c.L + kIxChunk - 1) / kIxChunk, c.T), kIxMarkThreads, 0, st>>>(p);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
      indexer_finish_kernel<<<c.T, kIxTopkThreads, 0, st>>>(p);
      e = cudaGetLastError();
    }
  }
  return e;
}

cudaError_t launch_indexer_scores(const IndexerCall& c, cudaStream_t st, int num_sms) {
  auto encode = c.encode;
  const int n_groups = (c.T + kIxQMax - 1) / kIxQMax;
  const size_t smem = (size_t)kIxStages * kIxStageBytes + 2 * (kIxQMax * kIxHeads) * 128 + 1024;
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  CUtensorMap kmap;
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)kIxD, (cuuint64_t)c.L};
    const cuuint64_t gstr[1] = {(cuuint64_t)kIxD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kIxKeys};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(c.keys), gdim, gstr, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int n_tiles = (c.L + kIxKeys - 1) / kIxKeys;
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  for (int g = 0; g < n_groups; ++g) {
    const int t0 = g * kIxQMax, tq = c.T - t0 < kIxQMax ? c.T - t0 : kIxQMax;
    CUtensorMap qmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)kIxD, (cuuint64_t)(tq * kIxHeads)};
    const cuuint64_t gstr[1] = {(cuuint64_t)kIxD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(tq * kIxHeads)};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<uint16_t*>(static_cast<const uint16_t*>(c.q) + (size_t)t0 * kIxHeads * kIxD), gdim, gstr,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    IxArgs p;
    p.T = tq;
    p.L = c.L;
    p.pos0 = c.pos0 + t0;
    p.w = c.w + (size_t)t0 * kIxHeads;
    p.scores = c.scores + (size_t)t0 * c.L;
    p.ls = c.L;
    p.hist = c.hist + ((size_t)t0 << 16);
    p.chist = c.chist + ((size_t)t0 << 11);
    p.status = c.status;
    p.wait_ns = c.wait_ns;
    indexer_scores_kernel<<<grid, kIxThreads, smem, st>>>(p, kmap, qmap);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace coli
